// LSE combine ("Chunk 66.0": the reduce half of the partial+reduce KV-split
// design) and the standalone ancestor-mask stage ("Chunk 66.1": mask-build).
//
// Combine: per query row, lse = ln sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) * O_s over the request's splits, written as bf16
// (round to nearest even) plus the fp32 lse.  One CTA per row; each of its 4
// warps owns 128 of the 512 output columns, each lane 4 of them (one float4
// load per split, coalesced 512 B per warp).  The warp reduces the split
// LSEs with shuffles.
#include "common.cuh"

namespace ddtree {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const VerifyArgs a) {
  const int g = blockIdx.x;
  const int b = g / a.rows_per_req;
  const int row = g - b * a.rows_per_req;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int first, count;
  request_slots(a, b, first, count);
  if (first + count > a.total_splits) {
    if (threadIdx.x == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
    count = max(0, a.total_splits - first);
  }
  const float* pl = a.partial_lse + row;
  const size_t lse_stride = (size_t)a.rows_per_req;

  float mx = -INFINITY;
  for (int s = lane; s < count; s += 32) mx = fmaxf(mx, pl[(size_t)(first + s) * lse_stride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

  float sum = 0.f;
  if (mx != -INFINITY) {
    for (int s = lane; s < count; s += 32) {
      float v = pl[(size_t)(first + s) * lse_stride];
      sum += (v == -INFINITY) ? 0.f : __expf(v - mx);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

  const int d = warp * 128 + lane * 4;
  const float* po = a.partial_o + (size_t)row * kLatent + d;
  const size_t o_stride = (size_t)a.rows_per_req * kLatent;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mx != -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < count; ++s) {
      float v = pl[(size_t)(first + s) * lse_stride];
      float w = (v == -INFINITY) ? 0.f : __expf(v - mx);
      float4 x = __ldg(reinterpret_cast<const float4*>(po + (size_t)(first + s) * o_stride));
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  }
  float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (size_t)g * kLatent + d) = pk;
  if (threadIdx.x == 0) a.lse[g] = sum > 0.f ? mx + logf(sum) : -INFINITY;
}

__global__ void ancestor_mask_kernel(const int32_t* parent, int T, uint64_t* anc, uint32_t* status) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < T) anc[(size_t)b * T + i] = ancestor_bits(parent + (size_t)b * T, i, T, status);
}

}  // namespace

cudaError_t launch_combine(const VerifyArgs& a, cudaStream_t stream) {
  combine_kernel<<<a.batch * a.rows_per_req, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ancestor_mask(const int32_t* parent, int batch, int n_nodes, uint64_t* anc,
                                 uint32_t* status, cudaStream_t stream) {
  ancestor_mask_kernel<<<batch, 64, 0, stream>>>(parent, n_nodes, anc, status);
  return cudaGetLastError();
}

}  // namespace ddtree
