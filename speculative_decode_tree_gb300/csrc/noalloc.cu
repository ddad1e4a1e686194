// Single-request verify attention that allocates nothing and takes no
// workspace argument.
//
// Who needs this: callers that cannot call cudaMalloc at the point where
// they run verify attention, for example code running under an allocator
// that forbids raw device allocations, a host thread inside a region where
// allocation would synchronise the device, or an integration with no place
// to keep a workspace buffer.  Such callers still own the inputs and the
// outputs; the split-KV partial results, which normally live in the caller's
// workspace, go to a scratch array that is part of this library's device
// image instead.
//
// The scratch is a file-scope device array of DDTREE_NOALLOC_SCRATCH_BYTES
// (8 MiB).  Every GPU that loads this library keeps those bytes reserved
// until the process exits.  All calls on a device share the one array and it
// keeps whatever the previous call left there: the status block at its start
// (status word and merge counters, 256 bytes) is cleared on the stream at the
// beginning of every call, and every partial
// result a call reads is written earlier in the same call.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on the array and corrupt each other's results; serialise them.
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace ddtree {
namespace {

constexpr size_t kScratchBytes = DDTREE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is only a stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DDTREE_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return DDTREE_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DDTREE_OK;
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Shrink the plan's split count until its partials fit the scratch array.
// Returns false when even one split per request does not fit.
bool fit_plan_to_scratch(ddtree_plan_t* p) {
  if (p->workspace_bytes <= (int64_t)kScratchBytes) return true;
  const int64_t rows = p->rows_per_req;
  const int64_t nkeys = p->max_keys;  // batch 1: the request's key count
  for (int64_t splits = p->total_splits - 1; splits >= 1; --splits) {
    int64_t chunk = round_up((nkeys + splits - 1) / splits, p->tile_keys);
    int64_t s = (nkeys + chunk - 1) / chunk;
    int64_t lse_bytes = round_up(s * rows * 4, 256);
    int64_t ws = 256 + lse_bytes + round_up(s * rows * (int64_t)kLatent * 2, 256);  // bf16 partial O
    if (ws <= (int64_t)kScratchBytes) {
      p->chunk_keys = (int32_t)chunk;
      p->total_splits = (int32_t)s;
      p->off_partial_lse = 256;
      p->off_partial_o = 256 + lse_bytes;
      p->workspace_bytes = ws;
      return true;
    }
  }
  return false;
}

inline bool aligned(const void* ptr, uintptr_t a) { return ((uintptr_t)ptr & (a - 1)) == 0; }

}  // namespace
}  // namespace ddtree

using namespace ddtree;

extern "C" int ddtree_verify_mla_noalloc(const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                                         const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                                         int prefix_len, const int32_t* tree_parent, int n_nodes,
                                         int n_heads, float sm_scale, ddtree_bf16_t* out, float* lse,
                                         struct CUstream_st* stream) {
  if (!q_latent || !q_rope || !kv_pool || !kv_indices || !tree_parent || !out || !lse)
    return DDTREE_EINVAL;
  if (!aligned(q_latent, 16) || !aligned(q_rope, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(kv_indices, 4) || !aligned(tree_parent, 4))
    return DDTREE_EINVAL;
  if (!isfinite(sm_scale)) return DDTREE_EINVAL;
  ddtree_plan_t plan;
  int32_t P = prefix_len;
  int rc = ddtree_verify_mla_plan(1, n_nodes, n_heads, &P, 0, &plan);
  if (rc != DDTREE_OK) return rc;
  if (!fit_plan_to_scratch(&plan)) return DDTREE_EWORKSPACE;  // needs more than the fixed scratch
  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_EUNSUPPORTED;
  }
  if (major != 10 || minor != 3) return DDTREE_EUNSUPPORTED;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != DDTREE_OK) return rc;

  VerifyArgs a;
  memset(&a, 0, sizeof(a));
  a.q_latent = q_latent;
  a.q_rope = q_rope;
  a.kv_pool = kv_pool;
  a.kv_indices = kv_indices;
  a.prefix_len_host = P;
  a.tree_parent = tree_parent;
  a.out = out;
  a.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.grid_done = reinterpret_cast<uint32_t*>(ws + 8);
  a.partial_lse = reinterpret_cast<float*>(ws + plan.off_partial_lse);
  a.partial_o = reinterpret_cast<uint16_t*>(ws + plan.off_partial_o);
  a.fused = plan.fused_combine;
  a.merge_depth = merge_depth_for(a.fused, plan.max_keys, plan.chunk_keys);
  a.wait_ns = 2000000000ull;
  a.pool_rows = 0;
  a.sm_scale = sm_scale;
  a.batch = 1;
  a.n_nodes = plan.n_nodes;
  a.n_heads = plan.n_heads;
  a.rows_per_req = plan.rows_per_req;
  a.tile_keys = plan.tile_keys;
  a.chunk_keys = plan.chunk_keys;
  a.total_splits = plan.total_splits;
  a.row_tile = plan.row_tile;
  a.row_tiles = plan.row_tiles;
  a.q_lat_stride = kLatent;
  a.q_rope_stride = kRope;

  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(a.status, 0, 256, s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  cudaError_t e = (plan.kernel == DDTREE_KERNEL_TC2)  ? launch_partial_tc2(a, s)
                  : (plan.kernel == DDTREE_KERNEL_TC) ? launch_partial_tc(a, s)
                                                      : launch_partial_simt(a, s);
  if (e == cudaSuccess && !a.fused) e = launch_combine(a, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}
