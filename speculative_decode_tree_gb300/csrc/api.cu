// Host side of the C ABI: planning (split heuristic), argument validation and
// the launch sequence.  No allocation, no host synchronisation (except the
// explicit status check), everything enqueued on the caller's stream.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace ddtree {
namespace {
constexpr int kMaxDevices = 64;
constexpr int64_t kStatusBytes = 256;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;
}  // namespace

// Cached SM count and compute capability of the current device.
int current_device_info(DevInfo* out) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return DDTREE_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev[d].valid) {
    DevInfo info{};
    if (cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess) {
      cudaGetLastError();
      return DDTREE_EUNSUPPORTED;
    }
    info.valid = true;
    g_dev[d] = info;
  }
  *out = g_dev[d];
  return DDTREE_OK;
}

namespace {

// Records a timing event; under stream capture it becomes an event-record
// node of the graph, so replays time the stages too.
cudaError_t record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  return cudaEventRecord(e, s);
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Tile geometry of each partial-kernel variant.
struct Geometry {
  int row_tile, tile_keys, waves;
};
Geometry geometry(int kernel) {
  if (kernel == DDTREE_KERNEL_TC || kernel == DDTREE_KERNEL_TC2) return Geometry{128, 128, 1};
  return Geometry{32, 32, 4};
}

// The tensor-core kernels work on 128-row tiles of 128 keys; below about one
// such tile's worth of (row, key) pairs the CUDA-core kernel is used.  Above
// it the cluster-of-four kernel runs, also for a single row tile (its second
// row tile then has no rows): with its merge in the same launch and its
// faster start it measured 27 us against the pair kernel's 42 us on a
// 128-row, 4k-key request.  The pair kernel stays available by request.
int choose_kernel(int kernel, int rows_per_req, int64_t total_keys) {
  if (kernel != DDTREE_KERNEL_AUTO) return kernel;
  if ((int64_t)rows_per_req * total_keys < 128 * 1024) return DDTREE_KERNEL_SIMT;
  return DDTREE_KERNEL_TC2;
}

// Bytes of one split's partial O rows (bf16) and LSEs (fp32).
inline int64_t partial_o_bytes(int64_t splits, int64_t rows) { return round_up(splits * rows * kLatent * 2, 256); }
inline int64_t partial_lse_bytes(int64_t splits, int64_t rows) { return round_up(splits * rows * 4, 256); }

// SMs the chosen kernel can keep busy at once on the current device.  A
// tensor-core work item is a cluster, and clusters are placed within one GPC,
// so a GPC whose SM count is not a multiple of the cluster size leaves SMs
// idle: the count is (clusters resident at once) x (cluster size).
int usable_sms(int kernel, int* out) {
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (kernel == DDTREE_KERNEL_SIMT || info.major != 10 || info.minor != 3) {
    *out = info.sms;
    return DDTREE_OK;
  }
  const int csize = kernel == DDTREE_KERNEL_TC2 ? 4 : 2;
  int clusters = 0;
  cudaError_t e = kernel == DDTREE_KERNEL_TC2 ? cluster_capacity_tc2(&clusters) : cluster_capacity_tc(&clusters);
  if (e != cudaSuccess || clusters < 1) {
    cudaGetLastError();
    return DDTREE_EUNSUPPORTED;
  }
  *out = std::min(info.sms, clusters * csize);
  return DDTREE_OK;
}

}  // namespace
}  // namespace ddtree

using namespace ddtree;

extern "C" int ddtree_verify_mla_plan_ex(int batch, int n_nodes, int n_heads,
                                         const int32_t* prefix_lens_host, int64_t pool_rows,
                                         int num_sms, int kernel, ddtree_plan_t* plan) {
  if (!plan || !prefix_lens_host) return DDTREE_EINVAL;
  if (batch < 1 || batch > DDTREE_MAX_BATCH) return DDTREE_EINVAL;
  if (n_nodes < 1 || n_nodes > DDTREE_MAX_NODES) return DDTREE_EINVAL;
  if (n_heads < 1 || n_heads > DDTREE_MAX_HEADS) return DDTREE_EINVAL;
  if (num_sms < 0 || num_sms > 4096) return DDTREE_EINVAL;
  if (kernel < DDTREE_KERNEL_AUTO || kernel > DDTREE_KERNEL_TC2) return DDTREE_EINVAL;
  int64_t total_keys = 0, max_keys = 0;
  for (int b = 0; b < batch; ++b) {
    if (prefix_lens_host[b] < 0 || prefix_lens_host[b] > (1 << 30)) return DDTREE_EINVAL;
    int64_t n = (int64_t)prefix_lens_host[b] + n_nodes;
    total_keys += n;
    max_keys = std::max(max_keys, n);
  }
  if (max_keys > INT32_MAX / 2) return DDTREE_EINVAL;

  ddtree_plan_t p;
  memset(&p, 0, sizeof(p));
  p.batch = batch;
  p.n_nodes = n_nodes;
  p.n_heads = n_heads;
  p.rows_per_req = n_nodes * n_heads;
  p.pool_rows = pool_rows;
  p.max_keys = (int32_t)max_keys;
  p.kernel = choose_kernel(kernel, p.rows_per_req, total_keys);
  const bool device_sized = num_sms == 0;
  if (num_sms == 0) {
    int rc = usable_sms(p.kernel, &num_sms);
    if (rc != DDTREE_OK) return rc;
  }
  p.num_sms = num_sms;
  Geometry g = geometry(p.kernel);
  p.row_tile = g.row_tile;
  p.tile_keys = g.tile_keys;
  p.row_tiles = (p.rows_per_req + g.row_tile - 1) / g.row_tile;

  // Split rule ("Chunk 66.1": the split count decides whether the SMs are
  // fed).  A work item is one row group x one key chunk; chunks are a whole
  // number of tiles.  A tensor-core work item is a cluster (2 CTAs for the
  // pair kernel, 4 for the cluster-of-four kernel covering two row tiles),
  // and the clusters the device holds at once make one wave.  The cluster
  // kernels take the shortest chunk whose work items -- counted after each
  // request's own rounding -- fit one wave; the CUDA-core kernel aims at a
  // few CTAs per SM.
  const int64_t ctas_per_item = p.kernel == DDTREE_KERNEL_TC2 ? 4 : (p.kernel == DDTREE_KERNEL_TC ? 2 : 1);
  const int64_t row_groups = p.kernel == DDTREE_KERNEL_TC2 ? (p.row_tiles + 1) / 2 : p.row_tiles;
  const int64_t target_items = std::max<int64_t>(1, (int64_t)g.waves * num_sms / ctas_per_item);
  auto items_for = [&](int64_t chunk) {
    int64_t n = 0;
    for (int b = 0; b < batch; ++b) n += ((int64_t)prefix_lens_host[b] + n_nodes + chunk - 1) / chunk;
    return n * row_groups;
  };
  const int64_t chunk_max = round_up(max_keys, g.tile_keys);
  int64_t chunk;
  if (p.kernel == DDTREE_KERNEL_SIMT) {
    const int64_t target_splits = std::max<int64_t>(1, (target_items + row_groups - 1) / row_groups);
    chunk = round_up(std::max<int64_t>((total_keys + target_splits - 1) / target_splits, g.tile_keys), g.tile_keys);
    chunk = std::min<int64_t>(chunk, chunk_max);
  } else {
    // Smallest k with items_for(k tiles) <= target (items fall as k grows).
    int64_t lo = 1, hi = chunk_max / g.tile_keys;
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (items_for(mid * g.tile_keys) <= target_items) hi = mid;
      else lo = mid + 1;
    }
    chunk = lo * g.tile_keys;
  }
  if (const char* env = getenv("DDTREE_CHUNK_KEYS")) {
    long v = strtol(env, nullptr, 10);
    if (v > 0) chunk = round_up(v, g.tile_keys);
  }
  p.chunk_keys = (int32_t)chunk;
  const int64_t splits = items_for(chunk) / row_groups;
  if (splits > INT32_MAX / 4) return DDTREE_EINVAL;
  p.total_splits = (int32_t)splits;
  // The cluster-of-four kernel merges the splits itself (no second launch)
  // when all of its clusters are resident at once on this device and a
  // request's splits fit one tile load of its merge.
  p.fused_combine = (p.kernel == DDTREE_KERNEL_TC2 && device_sized && items_for(chunk) <= target_items &&
                     merge_depth_for(1, (int)max_keys, (int)chunk) > 0)
                        ? 1
                        : 0;

  p.off_partial_lse = kStatusBytes;
  p.off_partial_o = p.off_partial_lse + partial_lse_bytes(splits, p.rows_per_req);
  p.workspace_bytes = p.off_partial_o + partial_o_bytes(splits, p.rows_per_req);
  *plan = p;
  return DDTREE_OK;
}

extern "C" int ddtree_verify_mla_plan(int batch, int n_nodes, int n_heads,
                                      const int32_t* prefix_lens_host, int64_t pool_rows,
                                      ddtree_plan_t* plan) {
  return ddtree_verify_mla_plan_ex(batch, n_nodes, n_heads, prefix_lens_host, pool_rows, 0,
                                   DDTREE_KERNEL_AUTO, plan);
}

extern "C" size_t ddtree_verify_mla_workspace_size(const ddtree_plan_t* plan) {
  return plan ? (size_t)plan->workspace_bytes : 0;
}

namespace {

int validate_plan(const ddtree_plan_t* p) {
  if (!p) return DDTREE_EINVAL;
  if (p->batch < 1 || p->batch > DDTREE_MAX_BATCH || p->n_nodes < 1 ||
      p->n_nodes > DDTREE_MAX_NODES || p->n_heads < 1 || p->n_heads > DDTREE_MAX_HEADS)
    return DDTREE_EINVAL;
  if (p->rows_per_req != p->n_nodes * p->n_heads) return DDTREE_EINVAL;
  if (p->kernel != DDTREE_KERNEL_SIMT && p->kernel != DDTREE_KERNEL_TC && p->kernel != DDTREE_KERNEL_TC2)
    return DDTREE_EINVAL;
  Geometry g = geometry(p->kernel);
  if (p->row_tile != g.row_tile || p->tile_keys != g.tile_keys) return DDTREE_EINVAL;
  if (p->row_tiles != (p->rows_per_req + g.row_tile - 1) / g.row_tile) return DDTREE_EINVAL;
  if (p->chunk_keys < p->tile_keys || p->chunk_keys % p->tile_keys) return DDTREE_EINVAL;
  if (p->total_splits < p->batch) return DDTREE_EINVAL;
  const int64_t lse_bytes = partial_lse_bytes(p->total_splits, p->rows_per_req);
  const int64_t o_bytes = partial_o_bytes(p->total_splits, p->rows_per_req);
  if (p->off_partial_lse != kStatusBytes || p->off_partial_o != kStatusBytes + lse_bytes ||
      p->workspace_bytes != p->off_partial_o + o_bytes)
    return DDTREE_EINVAL;
  if (p->fused_combine != 0 && (p->fused_combine != 1 || p->kernel != DDTREE_KERNEL_TC2 ||
                                merge_depth_for(1, p->max_keys, p->chunk_keys) == 0))
    return DDTREE_EINVAL;
  if (p->wait_limit_us < 0) return DDTREE_EINVAL;
  int ls = p->q_latent_row_stride, rs = p->q_rope_row_stride;
  if (ls != 0 && (ls < kLatent || ls % 8)) return DDTREE_EINVAL;
  if (rs != 0 && (rs < kRope || rs % 8)) return DDTREE_EINVAL;
  return DDTREE_OK;
}

int run(const ddtree_plan_t* p, const uint16_t* q_latent, const uint16_t* q_rope,
        const uint16_t* kv_pool, const int32_t* kv_indices, const int32_t* kv_indptr,
        const int32_t* prefix_lens, int32_t prefix_len_host, const int32_t* tree_parent,
        float sm_scale, uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
        cudaStream_t stream, cudaEvent_t const* ev = nullptr) {
  if (!q_latent || !q_rope || !kv_pool || !kv_indices || !tree_parent || !out || !lse || !workspace)
    return DDTREE_EINVAL;
  if (!aligned(q_latent, 16) || !aligned(q_rope, 16) || !aligned(kv_pool, 16) ||
      !aligned(out, 16) || !aligned(lse, 4) || !aligned(kv_indices, 4) ||
      !aligned(tree_parent, 4) || !aligned(workspace, 256))
    return DDTREE_EINVAL;
  if (!isfinite(sm_scale)) return DDTREE_EINVAL;
  if ((int64_t)workspace_bytes < p->workspace_bytes) return DDTREE_EWORKSPACE;
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (info.major != 10 || info.minor != 3) return DDTREE_EUNSUPPORTED;

  VerifyArgs a;
  memset(&a, 0, sizeof(a));
  a.q_latent = q_latent;
  a.q_rope = q_rope;
  a.kv_pool = kv_pool;
  a.kv_indices = kv_indices;
  a.kv_indptr = kv_indptr;
  a.prefix_lens = prefix_lens;
  a.prefix_len_host = prefix_len_host;
  a.tree_parent = tree_parent;
  a.out = out;
  a.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.grid_done = reinterpret_cast<uint32_t*>(ws + 8);
  a.partial_lse = reinterpret_cast<float*>(ws + p->off_partial_lse);
  a.partial_o = reinterpret_cast<uint16_t*>(ws + p->off_partial_o);
  a.fused = p->fused_combine;
  // Every request has at most ceil(max_keys / chunk) splits.
  a.merge_depth = merge_depth_for(a.fused, p->max_keys, p->chunk_keys);
  a.wait_ns = p->wait_limit_us > 0 ? (uint64_t)p->wait_limit_us * 1000ull : 2000000000ull;
  a.pool_rows = p->pool_rows;
  a.sm_scale = sm_scale;
  a.batch = p->batch;
  a.n_nodes = p->n_nodes;
  a.n_heads = p->n_heads;
  a.rows_per_req = p->rows_per_req;
  a.tile_keys = p->tile_keys;
  a.chunk_keys = p->chunk_keys;
  a.total_splits = p->total_splits;
  a.row_tile = p->row_tile;
  a.row_tiles = p->row_tiles;
  a.q_lat_stride = p->q_latent_row_stride ? p->q_latent_row_stride : kLatent;
  a.q_rope_stride = p->q_rope_row_stride ? p->q_rope_row_stride : kRope;

  if (cudaMemsetAsync(a.status, 0, 256, stream) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  cudaError_t e = cudaSuccess;
  if (ev && ev[0]) e = record_event(ev[0], stream);
  if (e == cudaSuccess)
    e = (p->kernel == DDTREE_KERNEL_TC2)  ? launch_partial_tc2(a, stream)
        : (p->kernel == DDTREE_KERNEL_TC) ? launch_partial_tc(a, stream)
                                          : launch_partial_simt(a, stream);
  if (e == cudaSuccess && ev && ev[1]) e = record_event(ev[1], stream);
  if (e == cudaSuccess && !a.fused) e = launch_combine(a, stream);
  if (e == cudaSuccess && ev && ev[2]) e = record_event(ev[2], stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}

}  // namespace

extern "C" int ddtree_verify_mla(const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                                 const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                                 int prefix_len, const int32_t* tree_parent, int n_nodes,
                                 int n_heads, float sm_scale, ddtree_bf16_t* out, float* lse,
                                 void* workspace, struct CUstream_st* stream) {
  ddtree_plan_t plan;
  int32_t P = prefix_len;
  int rc = ddtree_verify_mla_plan(1, n_nodes, n_heads, &P, 0, &plan);
  if (rc != DDTREE_OK) return rc;
  return run(&plan, q_latent, q_rope, kv_pool, kv_indices, nullptr, nullptr, P, tree_parent,
             sm_scale, out, lse, workspace, (size_t)plan.workspace_bytes, (cudaStream_t)stream);
}

extern "C" int ddtree_verify_mla_batched(const ddtree_plan_t* plan, const ddtree_bf16_t* q_latent,
                                         const ddtree_bf16_t* q_rope, const ddtree_bf16_t* kv_pool,
                                         const int32_t* kv_indices, const int32_t* kv_indptr,
                                         const int32_t* prefix_lens, const int32_t* tree_parent,
                                         float sm_scale, ddtree_bf16_t* out, float* lse,
                                         void* workspace, size_t workspace_bytes,
                                         struct CUstream_st* stream) {
  int rc = validate_plan(plan);
  if (rc != DDTREE_OK) return rc;
  if (!kv_indptr || !prefix_lens || !aligned(kv_indptr, 4) || !aligned(prefix_lens, 4))
    return DDTREE_EINVAL;
  return run(plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, 0, tree_parent,
             sm_scale, out, lse, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int ddtree_verify_mla_batched_timed(
    const ddtree_plan_t* plan, const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
    const ddtree_bf16_t* kv_pool, const int32_t* kv_indices, const int32_t* kv_indptr,
    const int32_t* prefix_lens, const int32_t* tree_parent, float sm_scale, ddtree_bf16_t* out,
    float* lse, void* workspace, size_t workspace_bytes, struct CUstream_st* stream,
    struct CUevent_st* const* stage_events) {
  int rc = validate_plan(plan);
  if (rc != DDTREE_OK) return rc;
  if (!kv_indptr || !prefix_lens || !aligned(kv_indptr, 4) || !aligned(prefix_lens, 4))
    return DDTREE_EINVAL;
  return run(plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, 0, tree_parent,
             sm_scale, out, lse, workspace, workspace_bytes, (cudaStream_t)stream,
             reinterpret_cast<cudaEvent_t const*>(stage_events));
}

extern "C" int ddtree_build_ancestor_mask(const int32_t* tree_parent, int batch, int n_nodes,
                                          uint64_t* anc_out, uint32_t* status,
                                          struct CUstream_st* stream) {
  if (!tree_parent || !anc_out || batch < 1 || batch > DDTREE_MAX_BATCH || n_nodes < 1 ||
      n_nodes > DDTREE_MAX_NODES || !aligned(tree_parent, 4) || !aligned(anc_out, 8) ||
      (status && !aligned(status, 4)))
    return DDTREE_EINVAL;
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (info.major != 10 || info.minor != 3) return DDTREE_EUNSUPPORTED;
  if (launch_ancestor_mask(tree_parent, batch, n_nodes, anc_out, status, (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}

extern "C" int ddtree_verify_mla_check(const void* workspace, struct CUstream_st* stream,
                                       uint32_t* host_status) {
  if (!workspace || !host_status || !aligned(workspace, 256)) return DDTREE_EINVAL;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  *host_status = v;
  return v ? DDTREE_EDEVICE_DATA : DDTREE_OK;
}

extern "C" const char* ddtree_status_str(int code) {
  switch (code) {
    case DDTREE_OK: return "ok";
    case DDTREE_EINVAL: return "invalid argument (null or misaligned pointer, or size out of range)";
    case DDTREE_EWORKSPACE: return "workspace smaller than the plan requires";
    case DDTREE_EUNSUPPORTED: return "no supported CUDA device (sm_103) is current";
    case DDTREE_ELAUNCH: return "kernel launch failed";
    case DDTREE_EDEVICE_DATA: return "device data error (bad index, parent or length)";
    case DDTREE_ECUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}
