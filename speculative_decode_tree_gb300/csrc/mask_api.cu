// Host side of the mask reader (include/ddtree_mask.h).
#include <string.h>

#include "common.cuh"
#include "../../include/ddtree_mask.h"

namespace ddtree {
namespace {
constexpr size_t kStatusBytes = 256;
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }
inline bool sizes_ok(int batch, int n_nodes) {
  return batch >= 1 && batch <= DDTREE_MAX_BATCH && n_nodes >= 1 && n_nodes <= DDTREE_MAX_NODES;
}
}  // namespace
}  // namespace ddtree

using namespace ddtree;

extern "C" size_t ddtree_tree_from_mask_workspace_size(int batch, int n_nodes) {
  if (!sizes_ok(batch, n_nodes)) return 0;
  return kStatusBytes + round256((size_t)batch * n_nodes * 8) + round256((size_t)batch * 4);
}

extern "C" int ddtree_tree_from_mask(int batch, int n_nodes, const uint8_t* custom_mask, const int64_t* mask_indptr,
                                     const int32_t* prefix_lens, int32_t* tree_parent, uint64_t* anc_bits,
                                     void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  if (!sizes_ok(batch, n_nodes)) return DDTREE_EINVAL;
  if (!custom_mask || !mask_indptr || !aligned(mask_indptr, 8) || !prefix_lens || !aligned(prefix_lens, 4) ||
      !tree_parent || !aligned(tree_parent, 4) || (anc_bits && !aligned(anc_bits, 8)) || !workspace ||
      !aligned(workspace, 256))
    return DDTREE_EINVAL;
  if (workspace_bytes < ddtree_tree_from_mask_workspace_size(batch, n_nodes)) return DDTREE_EWORKSPACE;
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (info.major != 10 || info.minor != 3) return DDTREE_EUNSUPPORTED;
  MaskArgs a;
  memset(&a, 0, sizeof(a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.mask = custom_mask;
  a.indptr = mask_indptr;
  a.prefix_lens = prefix_lens;
  a.parent = tree_parent;
  a.anc = anc_bits;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.rows = reinterpret_cast<uint64_t*>(ws + kStatusBytes);
  a.tickets = reinterpret_cast<uint32_t*>(ws + kStatusBytes + round256((size_t)batch * n_nodes * 8));
  a.batch = batch;
  a.n_nodes = n_nodes;
  a.num_sms = info.sms;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, ddtree_tree_from_mask_workspace_size(batch, n_nodes), s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  if (launch_mask(a, s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}
