// LSE combine ("Chunk 66.0": the reduce half of the partial+reduce KV-split
// design) and the standalone ancestor-mask stage ("Chunk 66.1": mask-build).
//
// Combine: per query row, lse = ln sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) * O_s over the request's splits, written as bf16
// (round to nearest even) plus the fp32 lse.  One 128-thread CTA per row:
// the block reduces the split LSEs (warp shuffles, then shared memory) and
// keeps the split weights in shared memory; each thread then owns 4 of the
// 512 output columns and streams the splits' float4 partials in batches of 16
// independent loads, so the L2-resident partials are read with enough loads
// in flight.
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kWeightSlots = 2048;  // splits per request whose weights stay in shared memory
constexpr int kBatch = 16;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) v = is_max ? fmaxf(v, red[i]) : v + red[i];
  return v;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const VerifyArgs a) {
  __shared__ float wts[kWeightSlots];
  __shared__ float red[kCombineThreads / 32];
  const int g = blockIdx.x;
  const int b = g / a.rows_per_req;
  const int row = g - b * a.rows_per_req;
  const int tid = threadIdx.x;
  int first, count;
  request_slots(a, b, first, count);
  if (first + count > a.total_splits) {
    if (tid == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
    count = max(0, a.total_splits - first);
  }
  const float* pl = a.partial_lse + (size_t)first * a.rows_per_req + row;
  const size_t lse_stride = (size_t)a.rows_per_req;

  float mx = -INFINITY;
  for (int s = tid; s < count; s += kCombineThreads) mx = fmaxf(mx, pl[(size_t)s * lse_stride]);
  mx = block_reduce(mx, true, red);
  float sum = 0.f;
  for (int s = tid; s < count; s += kCombineThreads) {
    const float v = pl[(size_t)s * lse_stride];
    const float w = (mx == -INFINITY || v == -INFINITY) ? 0.f : __expf(v - mx);
    if (s < kWeightSlots) wts[s] = w;
    sum += w;
  }
  sum = block_reduce(sum, false, red);  // its barriers also publish wts

  const int d = tid * 4;
  const size_t o_stride = (size_t)a.rows_per_req * kLatent;
  const float* po = a.partial_o + ((size_t)first * a.rows_per_req + row) * kLatent + d;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < count; s0 += kBatch) {
    float4 x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      x[j] = (s0 + j < count) ? __ldg(reinterpret_cast<const float4*>(po + (size_t)(s0 + j) * o_stride))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int s = s0 + j;
      if (s < count) {
        float w;
        if (s < kWeightSlots) {
          w = wts[s];
        } else {
          const float v = pl[(size_t)s * lse_stride];
          w = (mx == -INFINITY || v == -INFINITY) ? 0.f : __expf(v - mx);
        }
        acc.x = fmaf(w, x[j].x, acc.x);
        acc.y = fmaf(w, x[j].y, acc.y);
        acc.z = fmaf(w, x[j].z, acc.z);
        acc.w = fmaf(w, x[j].w, acc.w);
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (size_t)g * kLatent + d) = pk;
  if (tid == 0) a.lse[g] = sum > 0.f ? mx + logf(sum) : -INFINITY;
}

__global__ void ancestor_mask_kernel(const int32_t* parent, int T, uint64_t* anc, uint32_t* status) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < T) anc[(size_t)b * T + i] = ancestor_bits(parent + (size_t)b * T, i, T, status);
}

}  // namespace

cudaError_t launch_combine(const VerifyArgs& a, cudaStream_t stream) {
  combine_kernel<<<a.batch * a.rows_per_req, kCombineThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ancestor_mask(const int32_t* parent, int batch, int n_nodes, uint64_t* anc,
                                 uint32_t* status, cudaStream_t stream) {
  ancestor_mask_kernel<<<batch, 64, 0, stream>>>(parent, n_nodes, anc, status);
  return cudaGetLastError();
}

}  // namespace ddtree
