// Tensor-map encoding for the paged caches (see tensor_map.h).
#include "tensor_map.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "pagedattn.h"
#include "status.h"

namespace pa {
namespace {

constexpr int kTokensPerBlock = 16;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  return PA_OK;
}

int encode_cache_map(CUtensorMap* map, const void* cache, bool bf16, int num_blocks,
                     int num_kv_heads, int head_dim) {
  const cuuint64_t dims[2] = {cuuint64_t(head_dim),
                              cuuint64_t(num_blocks) * num_kv_heads * kTokensPerBlock};
  const cuuint64_t strides[1] = {cuuint64_t(head_dim) * 2};
  const cuuint32_t box[2] = {64, kTokensPerBlock};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PA_OK;
}

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
  CUtensorMap map;  // 64-byte aligned by its own declaration
};
constexpr int kMapCache = 256;
thread_local MapEntry t_maps[kMapCache];

}  // namespace

int cache_tensor_map(CUtensorMap* out, const void* cache, bool bf16, int num_blocks,
                     int num_kv_heads, int head_dim) {
  int rc = get_encoder();
  if (rc != PA_OK) return rc;
  const MapKey key{cache, num_blocks, num_kv_heads, head_dim, bf16};
  uint64_t h = reinterpret_cast<uintptr_t>(cache) >> 8;
  h ^= uint64_t(num_blocks) * 0x9E3779B97F4A7C15ull ^ uint64_t(num_kv_heads * 131 + head_dim);
  MapEntry& e = t_maps[(h ^ (h >> 17)) % kMapCache];
  if (!(e.key == key)) {
    rc = encode_cache_map(&e.map, cache, bf16, num_blocks, num_kv_heads, head_dim);
    if (rc != PA_OK) {
      e.key = MapKey{nullptr, 0, 0, 0, false};
      return rc;
    }
    e.key = key;
  }
  *out = e.map;
  return PA_OK;
}

int query_tensor_map(CUtensorMap* out, const void* q, bool bf16, int total_q, int num_q_heads,
                     int head_dim, int group, int rows) {
  int rc = get_encoder();
  if (rc != PA_OK) return rc;
  const cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(num_q_heads), cuuint64_t(total_q)};
  const cuuint64_t strides[2] = {cuuint64_t(head_dim) * 2, cuuint64_t(num_q_heads) * head_dim * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(rows / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(out, dt, 3, const_cast<void*>(q), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (query) failed (%d)", int(r));
  return PA_OK;
}

int output_tensor_map(CUtensorMap* out, void* o, bool bf16, int total_q, int num_q_heads,
                      int head_dim, int group, int rows) {
  int rc = get_encoder();
  if (rc != PA_OK) return rc;
  const cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(num_q_heads), cuuint64_t(total_q)};
  const cuuint64_t strides[2] = {cuuint64_t(head_dim) * 2, cuuint64_t(num_q_heads) * head_dim * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(rows / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(out, dt, 3, o, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", int(r));
  return PA_OK;
}

}  // namespace pa
