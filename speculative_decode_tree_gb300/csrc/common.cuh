// Shared device-side definitions of the DDTree verify-attention library.
#pragma once

#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ddtree_verify.h"

namespace ddtree {

constexpr int kLatent = DDTREE_LATENT_DIM;  // 512: value width
constexpr int kRope = DDTREE_ROPE_DIM;      // 64
constexpr int kRow = DDTREE_ROW_DIM;        // 576: key width
// The fused split merge loads a request's splits for two rows in one tile
// box (2 KB of shared memory per split) when there are at most this many.
constexpr int kMergeMaxSplits = 64;
// Splits per merge box for a plan (0: merge by warps instead).
inline int merge_depth_for(int fused, int max_keys, int chunk_keys) {
  if (!fused || chunk_keys <= 0) return 0;
  const long long d = ((long long)max_keys + chunk_keys - 1) / chunk_keys;
  return (d >= 1 && d <= kMergeMaxSplits) ? (int)d : 0;
}

// Everything a launch needs, resolved on the host from the plan and the
// caller's pointers.  Passed by value as a kernel parameter.
struct VerifyArgs {
  const uint16_t* q_latent;
  const uint16_t* q_rope;
  const uint16_t* kv_pool;
  const int32_t* kv_indices;
  const int32_t* kv_indptr;    // null: single request starting at index 0
  const int32_t* prefix_lens;  // null: single request of length prefix_len_host
  const int32_t* tree_parent;  // [B, T]
  uint16_t* out;
  float* lse;
  float* partial_lse;          // [total_splits, rows_per_req]
  uint16_t* partial_o;         // [total_splits, rows_per_req, 512] bf16
  uint32_t* status;            // workspace offset 0
  uint32_t* grid_done;         // workspace offset 8: CTAs finished (fused combine)
  int64_t pool_rows;           // <= 0: indices unchecked
  float sm_scale;
  int32_t prefix_len_host;
  int32_t batch, n_nodes, n_heads, rows_per_req;
  int32_t tile_keys, chunk_keys, total_splits, row_tile, row_tiles;
  int32_t q_lat_stride, q_rope_stride;
  int32_t fused;               // the partial kernel merges the splits itself
  int32_t merge_depth;         // fused merge by tile loads: splits per box (0: by warps)
  uint64_t wait_ns;            // bound of every wait inside the kernels
};

// One work item's request: which request a split slot belongs to, and the
// request's lengths as read on the device.
struct SplitLoc {
  int b;            // request
  int s;            // split within the request
  int P;            // prefix length
  int nkeys;        // P + T
  int ns;           // splits of the request
  int64_t idx_base; // first kv_indices entry of the request
};

__device__ __forceinline__ int dev_prefix_len(const VerifyArgs& a, int b) {
  return a.prefix_lens ? __ldg(a.prefix_lens + b) : a.prefix_len_host;
}

// Maps split slot w to (request, split).  Slots are laid out request by
// request: request b owns ceil((P_b+T)/chunk) consecutive slots.  Returns
// false (and flags BAD_LENGTH when lengths are inconsistent) for slots past
// the last request; the plan sizes total_splits for the longest lengths.
__device__ __forceinline__ bool locate_split(const VerifyArgs& a, int w, SplitLoc& loc) {
  int acc = 0;
  for (int r = 0; r < a.batch; ++r) {
    // The request's index range is loaded together with its length (a load
    // behind the length test would wait for the length first).
    int P = dev_prefix_len(a, r);
    const auto i0 = a.kv_indptr ? __ldg(a.kv_indptr + r) : 0;
    const auto i1 = a.kv_indptr ? __ldg(a.kv_indptr + r + 1) : 0;
    if (P < 0 || P > INT32_MAX - 2 * DDTREE_MAX_NODES) {
      atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
      return false;
    }
    int n = P + a.n_nodes;
    int ns = (int)(((int64_t)n + a.chunk_keys - 1) / a.chunk_keys);
    if (w < acc + ns) {
      loc.b = r;
      loc.s = w - acc;
      loc.P = P;
      loc.nkeys = n;
      loc.ns = ns;
      loc.idx_base = (int64_t)i0;
      if (a.kv_indptr && i1 - i0 != n) {
        atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
        return false;
      }
      if (acc + ns > a.total_splits) {  // longer than planned: no slot
        atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
        return false;
      }
      return true;
    }
    acc += ns;
  }
  return false;
}

// First slot and split count of request b (for the combine stage).
// Split counts are taken in 64 bits: P + T + chunk can pass INT32_MAX when
// one split covers nearly all keys.
__device__ __forceinline__ void request_slots(const VerifyArgs& a, int b, int& first, int& count) {
  int64_t acc = 0;
  for (int r = 0; r < b; ++r) {
    const int64_t P = max(dev_prefix_len(a, r), 0);
    acc += (P + a.n_nodes + a.chunk_keys - 1) / a.chunk_keys;
  }
  const int64_t P = max(dev_prefix_len(a, b), 0);
  first = (int)(acc < (int64_t)INT32_MAX ? acc : (int64_t)INT32_MAX);
  count = (int)((P + a.n_nodes + a.chunk_keys - 1) / a.chunk_keys);
}

// Ancestor set of node i as a bitmask: bit j set when j is i or one of its
// ancestors.  parent[i] must be -1 or an earlier node; the walk stops at the
// first parent that is not, and flags BAD_PARENT.  At most T steps because
// every accepted parent is strictly smaller than its child.
__device__ __forceinline__ uint64_t ancestor_bits(const int32_t* parent, int i, int T,
                                                  uint32_t* status) {
  uint64_t bits = 0;
  int a = i;
  for (int step = 0; step < T && a >= 0; ++step) {
    bits |= 1ull << a;
    int p = __ldg(parent + a);
    if (p < -1 || p >= a) {
      if (status) atomicOr(status, DDTREE_ST_BAD_PARENT);
      break;
    }
    a = p;
  }
  return bits;
}

// The same walk over a parent array already staged in shared memory (one
// coalesced load instead of a chain of dependent global loads per node).
__device__ __forceinline__ uint64_t ancestor_bits_smem(const int32_t* parent, int i, int T, uint32_t* status) {
  uint64_t bits = 0;
  int a = i;
  for (int step = 0; step < T && a >= 0; ++step) {
    bits |= 1ull << a;
    const int p = parent[a];
    if (p < -1 || p >= a) {
      if (status) atomicOr(status, DDTREE_ST_BAD_PARENT);
      break;
    }
    a = p;
  }
  return bits;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Cached SM count and compute capability of the current device (api.cu).
struct DevInfo {
  bool valid;
  int sms, major, minor;
};
int current_device_info(DevInfo* out);

// Everything the acceptance launch needs (see include/ddtree_accept.h).
struct AcceptArgs {
  const uint16_t* logits;   // [B, T+1, V] bf16
  const int32_t* draft;     // [B, T]
  const int32_t* parent;    // [B, T]
  const int32_t* kv_indices;
  const int32_t* kv_indptr;    // [B+1]
  const int32_t* prefix_lens;  // [B]
  uint64_t* keys;           // workspace: [B, T+1] argmax keys, zeroed by the launch sequence
  uint32_t* tickets;        // workspace: [B] CTAs done per request, zeroed likewise
  int32_t* accept_len;      // [B]
  int32_t* next_token;      // [B]
  int32_t* accepted_nodes;  // [B, T]
  int32_t* commit_indices;  // [B, T]
  int32_t* freed_indices;   // [B, T]
  uint32_t* status;         // workspace offset 0
  int batch, n_nodes, vocab, num_sms;
};

// Everything the relocation launches need (see include/ddtree_relocate.h).
struct RelocateArgs {
  uint16_t* pool;            // [pool_rows, 576] bf16, updated in place
  int32_t* indices;          // [total_rows], updated in place
  const int32_t* indptr;     // [batch+1]
  const int32_t* dest;       // [batch]
  int32_t* old_indices;      // [total_rows] or null
  uint32_t* bitmap;          // workspace: one bit per pool row, zeroed by the launch sequence
  uint32_t* status;          // workspace offset 0
  int64_t pool_rows, total_rows;
  int batch;
};

// Everything the mask reader needs (see include/ddtree_mask.h).
struct MaskArgs {
  const uint8_t* mask;
  const int64_t* indptr;     // [batch+1] element offsets
  const int32_t* prefix_lens;
  int32_t* parent;           // [batch, n_nodes]
  uint64_t* anc;             // [batch, n_nodes] or null
  uint64_t* rows;            // workspace: [batch, n_nodes] visible-node bits
  uint32_t* tickets;         // workspace: [batch]
  uint32_t* status;          // workspace offset 0
  int batch, n_nodes, num_sms;
};

// ---- launchers (one per .cu file) ----
cudaError_t launch_mask(const MaskArgs& a, cudaStream_t stream);
cudaError_t launch_relocate(const RelocateArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t stream);
cudaError_t launch_partial_simt(const VerifyArgs& a, cudaStream_t stream);
cudaError_t launch_partial_tc(const VerifyArgs& a, cudaStream_t stream);
cudaError_t launch_partial_tc2(const VerifyArgs& a, cudaStream_t stream);
cudaError_t cluster_capacity_tc(int* clusters);
cudaError_t cluster_capacity_tc2(int* clusters);
cudaError_t launch_combine(const VerifyArgs& a, cudaStream_t stream);
cudaError_t launch_ancestor_mask(const int32_t* parent, int batch, int n_nodes, uint64_t* anc,
                                 uint32_t* status, cudaStream_t stream);

}  // namespace ddtree
