// Host side of the relocation entry points (include/ddtree_relocate.h).
#include <string.h>

#include "common.cuh"
#include "../../include/ddtree_relocate.h"

namespace ddtree {
namespace {
constexpr size_t kStatusBytes = 256;
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline size_t bitmap_bytes(int64_t pool_rows) { return ((size_t)((pool_rows + 31) / 32) * 4 + 255) / 256 * 256; }
}  // namespace
}  // namespace ddtree

using namespace ddtree;

extern "C" size_t ddtree_relocate_kv_workspace_size(int64_t pool_rows) {
  if (pool_rows < 1 || pool_rows > INT32_MAX) return 0;
  return kStatusBytes + bitmap_bytes(pool_rows);
}

extern "C" int ddtree_relocate_kv(int batch, int64_t total_rows, ddtree_bf16_t* kv_pool, int64_t pool_rows,
                                  int32_t* kv_indices, const int32_t* kv_indptr, const int32_t* dest_base,
                                  int32_t* old_indices, void* workspace, size_t workspace_bytes,
                                  struct CUstream_st* stream) {
  if (batch < 1 || batch > DDTREE_MAX_BATCH || pool_rows < 1 || pool_rows > INT32_MAX || total_rows < 0 ||
      total_rows > pool_rows)
    return DDTREE_EINVAL;
  if (!kv_pool || !aligned(kv_pool, 16) || !kv_indices || !aligned(kv_indices, 4) || !kv_indptr ||
      !aligned(kv_indptr, 4) || !dest_base || !aligned(dest_base, 4) || (old_indices && !aligned(old_indices, 4)) ||
      !workspace || !aligned(workspace, 256))
    return DDTREE_EINVAL;
  if (workspace_bytes < ddtree_relocate_kv_workspace_size(pool_rows)) return DDTREE_EWORKSPACE;
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (info.major != 10 || info.minor != 3) return DDTREE_EUNSUPPORTED;

  RelocateArgs a;
  memset(&a, 0, sizeof(a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.pool = kv_pool;
  a.indices = kv_indices;
  a.indptr = kv_indptr;
  a.dest = dest_base;
  a.old_indices = old_indices;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.bitmap = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  a.pool_rows = pool_rows;
  a.total_rows = total_rows;
  a.batch = batch;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, ddtree_relocate_kv_workspace_size(pool_rows), s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  if (launch_relocate(a, info.sms, s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}
