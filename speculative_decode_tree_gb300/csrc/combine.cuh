// The log-sum-exp merge of the split partials ("Chunk 66.0": the reduce half
// of the KV-split partial + reduce design), as a warp-level unit of work used
// by the standalone combine kernel and by the partial kernel that merges its
// own splits.
//
// One unit = one query row x 64 of the 512 output columns; lane l owns
// columns 2l, 2l+1 (one 4-byte bf16 pair per split, so a warp's loads of a
// split are one coalesced 128-byte line).  Over the request's splits s:
//     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
// taken in one pass with a running maximum; a batch holds every split a
// one-wave plan makes, so the merge is a single round of independent loads.
#pragma once

#include "common.cuh"

namespace ddtree {

constexpr int kCombineCols = 64;           // output columns per unit
constexpr int kCombineUnitsPerRow = kLatent / kCombineCols;
constexpr int kCombineBatch = 36;          // splits loaded per round

// Units of a call: every (request, row, 64-column part).
__device__ __forceinline__ int combine_units(const VerifyArgs& a) {
  return a.batch * a.rows_per_req * kCombineUnitsPerRow;
}

// Merges unit u.  `zero` writes a zero row and -inf LSE instead (used when
// the partials cannot be trusted, e.g. after a timed-out wait).
__device__ __forceinline__ void combine_unit(const VerifyArgs& a, int u, int lane, bool zero) {
  const int part = u % kCombineUnitsPerRow;
  const int g = u / kCombineUnitsPerRow;  // global query row (request-major)
  const int b = g / a.rows_per_req;
  const int row = g - b * a.rows_per_req;
  const int d = part * kCombineCols + 2 * lane;
  int first = 0, count = 0;
  if (!zero) {
    request_slots(a, b, first, count);
    if (first + count > a.total_splits) {
      if (lane == 0 && part == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
      count = max(0, a.total_splits - first);
    }
  }
  const size_t rows = (size_t)a.rows_per_req;
  const float* pl = a.partial_lse + (size_t)first * rows + row;
  const uint16_t* po = a.partial_o + ((size_t)first * rows + row) * kLatent + d;
  const size_t o_stride = rows * kLatent;

  float m = -INFINITY, l = 0.f, acc0 = 0.f, acc1 = 0.f;
  for (int s0 = 0; s0 < count; s0 += kCombineBatch) {
    float ls[kCombineBatch];
    uint32_t x[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const bool in = s0 + j < count;
      // L2-coherent loads: in the fused form the partials were written by
      // other CTAs of the same launch.
      ls[j] = in ? __ldcg(pl + (size_t)(s0 + j) * rows) : -INFINITY;
      x[j] = in ? __ldcg(reinterpret_cast<const uint32_t*>(po + (size_t)(s0 + j) * o_stride)) : 0u;
    }
    float bm = m;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) bm = fmaxf(bm, ls[j]);
    if (bm == -INFINITY) continue;  // nothing attended so far
    const float scale = (m == -INFINITY) ? 0.f : __expf(m - bm);
    l *= scale;
    acc0 *= scale;
    acc1 *= scale;
    m = bm;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const float w = (ls[j] == -INFINITY) ? 0.f : __expf(ls[j] - m);
      l += w;
      acc0 = fmaf(w, bf16_lo(x[j]), acc0);
      acc1 = fmaf(w, bf16_hi(x[j]), acc1);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  *reinterpret_cast<__nv_bfloat162*>(a.out + (size_t)g * kLatent + d) = __floats2bfloat162_rn(acc0 * inv, acc1 * inv);
  if (part == 0 && lane == 0) a.lse[g] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace ddtree
