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
// A batch's LSEs are spread over the lanes (two per lane) and each split's
// weight is computed once and broadcast by a shuffle.
#pragma once

#include "common.cuh"

namespace ddtree {

constexpr int kCombineCols = 64;           // output columns per unit
constexpr int kCombineUnitsPerRow = kLatent / kCombineCols;
constexpr int kCombineBatch = 36;          // splits loaded per round (<= 64: two LSEs per lane)

// Units of a call: every (request, row, 64-column part).
__device__ __forceinline__ int combine_units(const VerifyArgs& a) {
  return a.batch * a.rows_per_req * kCombineUnitsPerRow;
}

// The split slots [first, first + count) of unit u's request (inconsistent
// lengths are flagged and clipped to the partial storage).
__device__ __forceinline__ void combine_slots(const VerifyArgs& a, int u, int lane, int& first, int& count) {
  const int g = u / kCombineUnitsPerRow;
  const int b = g / a.rows_per_req;
  request_slots(a, b, first, count);
  if (first + count > a.total_splits) {
    if (lane == 0 && u % kCombineUnitsPerRow == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
    count = max(0, a.total_splits - first);
  }
}

// Merges unit u over the split slots [first, first + count).  count == 0
// writes a zero row and -inf LSE (also used when the partials cannot be
// trusted, e.g. after a timed-out wait).
__device__ __forceinline__ void combine_unit(const VerifyArgs& a, int u, int lane, int first, int count) {
  const int part = u % kCombineUnitsPerRow;
  const int g = u / kCombineUnitsPerRow;  // global query row (request-major)
  const int row = g - (g / a.rows_per_req) * a.rows_per_req;
  const int d = part * kCombineCols + 2 * lane;
  const size_t rows = (size_t)a.rows_per_req;
  const float* pl = a.partial_lse + (size_t)first * rows + row;
  const uint32_t* po = reinterpret_cast<const uint32_t*>(a.partial_o + ((size_t)first * rows + row) * kLatent + d);
  const size_t o_stride = rows * kLatent / 2;  // in bf16 pairs

  float m = -INFINITY, lp = 0.f, acc0 = 0.f, acc1 = 0.f;  // lp: this lane's share of l
  for (int s0 = 0; s0 < count; s0 += kCombineBatch) {
    const int nb = min(count - s0, kCombineBatch);
    // Every load is issued unconditionally (split index clamped into the
    // batch), so all of them are in flight at once; the batch bound is
    // applied where the values are used.  (A load under a condition feeding
    // a select waits for each load in turn.)  L2-coherent loads: in the
    // fused form the partials were written by other CTAs of the same launch.
    uint32_t x[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) x[j] = __ldcg(po + (size_t)(s0 + min(j, nb - 1)) * o_stride);
    // Lane j holds the LSE of splits s0 + j and s0 + 32 + j.
    const float la = __ldcg(pl + (size_t)(s0 + min(lane, nb - 1)) * rows);
    const float lb = __ldcg(pl + (size_t)(s0 + min(lane + 32, nb - 1)) * rows);
    const float va = lane < nb ? la : -INFINITY, vb = lane + 32 < nb ? lb : -INFINITY;
    float bm = fmaxf(va, vb);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    bm = fmaxf(bm, m);
    if (bm == -INFINITY) continue;  // nothing attended so far
    const float scale = (m == -INFINITY) ? 0.f : __expf(m - bm);
    m = bm;
    const float wa = va == -INFINITY ? 0.f : __expf(va - m);
    const float wb = vb == -INFINITY ? 0.f : __expf(vb - m);
    lp = lp * scale + wa + wb;
    acc0 *= scale;
    acc1 *= scale;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const float w = j < nb ? __shfl_sync(0xffffffffu, j < 32 ? wa : wb, j & 31) : 0.f;
      acc0 = fmaf(w, bf16_lo(x[j]), acc0);
      acc1 = fmaf(w, bf16_hi(x[j]), acc1);
    }
  }
  float l = lp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  *reinterpret_cast<__nv_bfloat162*>(a.out + (size_t)g * kLatent + d) = __floats2bfloat162_rn(acc0 * inv, acc1 * inv);
  if (part == 0 && lane == 0) a.lse[g] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace ddtree
