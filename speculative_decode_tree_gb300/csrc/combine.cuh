// The log-sum-exp merge of the split partials ("Chunk 66.0": the reduce half
// of the KV-split partial + reduce design), as a warp-level unit of work used
// by the standalone combine kernel and by the partial kernel that merges its
// own splits.
//
// One unit = one query row x 128 of the 512 output columns; lane l owns
// columns 4l .. 4l+3.  Over the request's splits s:
//     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
// taken in one pass with a running maximum so that every load is independent
// (all of a batch's split LSEs and partial rows are in flight together).
#pragma once

#include "common.cuh"

namespace ddtree {

constexpr int kCombineCols = 128;          // output columns per unit
constexpr int kCombineUnitsPerRow = kLatent / kCombineCols;
constexpr int kCombineBatch = 12;          // splits loaded per batch

// Units of a call: every (request, row, column quarter).
__device__ __forceinline__ int combine_units(const VerifyArgs& a) {
  return a.batch * a.rows_per_req * kCombineUnitsPerRow;
}

__device__ __forceinline__ void store_bf16x4(uint16_t* dst, float x, float y, float z, float w) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(x, y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(z, w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = pk;
}

// Merges unit u.  `zero` writes a zero row and -inf LSE instead (used when
// the partials cannot be trusted, e.g. after a timed-out wait).
__device__ __forceinline__ void combine_unit(const VerifyArgs& a, int u, int lane, bool zero) {
  const int quarter = u % kCombineUnitsPerRow;
  const int g = u / kCombineUnitsPerRow;  // global query row (request-major)
  const int b = g / a.rows_per_req;
  const int row = g - b * a.rows_per_req;
  const int d = quarter * kCombineCols + 4 * lane;
  int first = 0, count = 0;
  if (!zero) {
    request_slots(a, b, first, count);
    if (first + count > a.total_splits) {
      if (lane == 0 && quarter == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
      count = max(0, a.total_splits - first);
    }
  }
  const size_t rows = (size_t)a.rows_per_req;
  const float* pl = a.partial_lse + (size_t)first * rows + row;
  const uint16_t* po = a.partial_o + ((size_t)first * rows + row) * kLatent + d;
  const size_t o_stride = rows * kLatent;

  float m = -INFINITY, l = 0.f;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
  for (int s0 = 0; s0 < count; s0 += kCombineBatch) {
    float ls[kCombineBatch];
    uint2 x[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const bool in = s0 + j < count;
      ls[j] = in ? __ldg(pl + (size_t)(s0 + j) * rows) : -INFINITY;
      x[j] = in ? __ldg(reinterpret_cast<const uint2*>(po + (size_t)(s0 + j) * o_stride)) : make_uint2(0u, 0u);
    }
    float bm = m;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) bm = fmaxf(bm, ls[j]);
    if (bm == -INFINITY) continue;  // nothing attended so far
    const float scale = (m == -INFINITY) ? 0.f : __expf(m - bm);
    l *= scale;
    acc0 *= scale; acc1 *= scale; acc2 *= scale; acc3 *= scale;
    m = bm;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const float w = (ls[j] == -INFINITY) ? 0.f : __expf(ls[j] - m);
      l += w;
      acc0 = fmaf(w, bf16_lo(x[j].x), acc0);
      acc1 = fmaf(w, bf16_hi(x[j].x), acc1);
      acc2 = fmaf(w, bf16_lo(x[j].y), acc2);
      acc3 = fmaf(w, bf16_hi(x[j].y), acc3);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  store_bf16x4(a.out + (size_t)g * kLatent + d, acc0 * inv, acc1 * inv, acc2 * inv, acc3 * inv);
  if (quarter == 0 && lane == 0) a.lse[g] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace ddtree
