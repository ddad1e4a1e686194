// Tier-1 KV relocation ("Chunk 66.1": live relocation of a request's rows into
// one contiguous region of the token-granular pool) and its checks.
//
// Three launches, each over the batch's rows (one thread or one warp per row):
//   mark  - every destination row sets its bit in a pool-sized bitmap; a bit
//           already set means two destination regions overlap;
//   check - every source index must lie in the pool and must not have its bit
//           set (a destination would overwrite a row the batch reads);
//   copy  - only if no check failed: one warp per row copies the 1152-byte row
//           with 16-byte loads and stores (two rows in flight per warp) and
//           rewrites the row's index.  HBM-bound: each row is read once and
//           written once.
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int kRowVec = kRow * 2 / 16;  // 72 sixteen-byte pieces per row

// Request of global row g: the last b with indptr[b] <= g (indptr ascending).
__device__ __forceinline__ int request_of(const int32_t* indptr, int batch, int64_t g) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(indptr + mid) <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void mark_kernel(RelocateArgs a) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g == 0) {
    // The layout itself: ascending offsets that end at total_rows.
    bool ok = __ldg(a.indptr) == 0 && (int64_t)__ldg(a.indptr + a.batch) == a.total_rows;
    for (int b = 0; b < a.batch && ok; ++b) ok = __ldg(a.indptr + b + 1) >= __ldg(a.indptr + b);
    if (!ok) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
  }
  int64_t row = -1;
  if (g < a.total_rows) {
    const int b = request_of(a.indptr, a.batch, g);
    const int64_t n = (int64_t)__ldg(a.indptr + b + 1) - __ldg(a.indptr + b);
    const int64_t k = g - __ldg(a.indptr + b);
    const int64_t d = __ldg(a.dest + b);
    if (k >= 0 && k < n) {  // else: inconsistent offsets, flagged above
      if (d < 0 || d + n > a.pool_rows) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
      else row = d + k;
    }
  }
  // Destination rows are consecutive within a request, so a warp's rows
  // share one or two bitmap words: one atomic per word, not per row.
  const uint64_t word = row < 0 ? ~0ull : (uint64_t)(row >> 5);
  const uint32_t bit = row < 0 ? 0u : 1u << (row & 31);
  const unsigned peers = __match_any_sync(0xffffffffu, word);
  const uint32_t bits = __reduce_or_sync(peers, bit);
  if (row >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) {
    // Two lanes with the same row (regions of two requests overlapping
    // inside this warp) leave fewer bits than lanes.
    if ((atomicOr(a.bitmap + word, bits) & bits) || __popc(bits) != __popc(peers))
      atomicOr(a.status, DDTREE_ST_OVERLAP);
  }
}

__global__ void check_kernel(RelocateArgs a) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= a.total_rows) return;
  const int64_t src = __ldg(a.indices + g);
  if (src < 0 || src >= a.pool_rows) {
    atomicOr(a.status, DDTREE_ST_BAD_INDEX);
    return;
  }
  if (__ldcg(a.bitmap + (src >> 5)) & (1u << (src & 31))) atomicOr(a.status, DDTREE_ST_OVERLAP);
}

__global__ void __launch_bounds__(256) copy_kernel(RelocateArgs a) {
  const bool ok = __ldcg(a.status) == 0;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t g0 = 2 * warp; g0 < a.total_rows; g0 += 2 * nwarps) {
    int32_t src[2];
    int64_t dst[2];
    bool have[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t g = g0 + r;
      have[r] = g < a.total_rows;
      src[r] = have[r] ? __ldg(a.indices + g) : 0;
      if (have[r]) {
        const int b = request_of(a.indptr, a.batch, g);
        dst[r] = (int64_t)__ldg(a.dest + b) + (g - __ldg(a.indptr + b));
      }
    }
    if (ok) {
      uint4 v[2][3];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint4* s = reinterpret_cast<const uint4*>(a.pool + (int64_t)src[r] * kRow);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int p = lane + 32 * j;
          if (have[r] && p < kRowVec) v[r][j] = __ldcs(s + p);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint4* d = reinterpret_cast<uint4*>(a.pool + dst[r] * kRow);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int p = lane + 32 * j;
          if (have[r] && p < kRowVec) d[p] = v[r][j];
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (!have[r]) continue;
        if (a.old_indices) a.old_indices[g0 + r] = src[r];
        if (ok) a.indices[g0 + r] = (int32_t)dst[r];
      }
    }
  }
}

}  // namespace

cudaError_t launch_relocate(const RelocateArgs& a, int num_sms, cudaStream_t stream) {
  if (a.total_rows > 0) {
    const unsigned blocks = (unsigned)((a.total_rows + 255) / 256);
    mark_kernel<<<blocks, 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    check_kernel<<<blocks, 256, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    mark_kernel<<<1, 32, 0, stream>>>(a);  // still validates the offsets
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t warps_needed = (a.total_rows + 1) / 2;
  const int64_t blocks = std::min<int64_t>((warps_needed + 7) / 8, (int64_t)num_sms * 8);
  copy_kernel<<<(unsigned)std::max<int64_t>(blocks, 1), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ddtree
