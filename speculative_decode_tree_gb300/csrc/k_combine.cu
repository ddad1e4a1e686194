// LSE combine ("Chunk 66.0": the reduce half of the partial+reduce KV-split
// design) and the standalone ancestor-mask stage ("Chunk 66.1": mask-build).
//
// Combine: per query row, lse = ln sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) * O_s over the request's splits, written as bf16
// (round to nearest even) plus the fp32 lse.  One 128-thread CTA per row;
// each thread owns 4 of the 512 output columns and makes a single pass over
// the splits with a running maximum (rescaling its partial sums when the
// maximum grows), so every load is independent of the others: the split
// LSEs (the same for all threads, served by L1) and the float4 partials are
// issued in batches of 16 and the whole combine costs a few memory round
// trips rather than a reduction tree.
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kBatch = 16;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const VerifyArgs a) {
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
  const int d = tid * 4;
  const size_t o_stride = (size_t)a.rows_per_req * kLatent;
  const float* po = a.partial_o + ((size_t)first * a.rows_per_req + row) * kLatent + d;

  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < count; s0 += kBatch) {
    float4 x[kBatch];
    float ls[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool in = s0 + j < count;
      ls[j] = in ? __ldg(pl + (size_t)(s0 + j) * lse_stride) : -INFINITY;
      x[j] = in ? __ldg(reinterpret_cast<const float4*>(po + (size_t)(s0 + j) * o_stride))
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float bm = m;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) bm = fmaxf(bm, ls[j]);
    if (bm == -INFINITY) continue;  // nothing attended so far
    const float scale = (m == -INFINITY) ? 0.f : __expf(m - bm);
    l *= scale;
    acc.x *= scale; acc.y *= scale; acc.z *= scale; acc.w *= scale;
    m = bm;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = (ls[j] == -INFINITY) ? 0.f : __expf(ls[j] - m);
      l += w;
      acc.x = fmaf(w, x[j].x, acc.x);
      acc.y = fmaf(w, x[j].y, acc.y);
      acc.z = fmaf(w, x[j].z, acc.z);
      acc.w = fmaf(w, x[j].w, acc.w);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (size_t)g * kLatent + d) = pk;
  if (tid == 0) a.lse[g] = l > 0.f ? m + logf(l) : -INFINITY;
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
