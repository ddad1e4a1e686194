// LSE combine ("Chunk 66.0": the reduce half of the partial+reduce KV-split
// design) and the standalone ancestor-mask stage ("Chunk 66.1": mask-build).
//
// Combine: per query row, lse = ln sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) * O_s over the request's splits, written as bf16
// (round to nearest even) plus the fp32 lse.  One warp per (row, 64 output
// columns); the merge itself is combine_unit (combine.cuh), shared with the
// partial kernel that merges its own splits.
#include "combine.cuh"

namespace ddtree {
namespace {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(const VerifyArgs a) {
  const int u = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (u >= combine_units(a)) return;
  int first, count;
  combine_slots(a, u, threadIdx.x & 31, first, count);
  combine_unit(a, u, threadIdx.x & 31, first, count);
}

__global__ void ancestor_mask_kernel(const int32_t* parent, int T, uint64_t* anc, uint32_t* status) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < T) anc[(size_t)b * T + i] = ancestor_bits(parent + (size_t)b * T, i, T, status);
}

}  // namespace

cudaError_t launch_combine(const VerifyArgs& a, cudaStream_t stream) {
  const int units = a.batch * a.rows_per_req * kCombineUnitsPerRow;
  combine_kernel<<<(units + kCombineWarps - 1) / kCombineWarps, 32 * kCombineWarps, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ancestor_mask(const int32_t* parent, int batch, int n_nodes, uint64_t* anc,
                                 uint32_t* status, cudaStream_t stream) {
  ancestor_mask_kernel<<<batch, 64, 0, stream>>>(parent, n_nodes, anc, status);
  return cudaGetLastError();
}

}  // namespace ddtree
