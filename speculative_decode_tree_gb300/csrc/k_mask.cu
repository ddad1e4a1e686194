// Flattened custom tree mask -> parent array and ancestor bits
// ("Chunk 66.1": the host mask-build the serving framework does; this reads
// its output on the device instead of taking a parent array).
//
// One launch, grid = (T rows, B requests, S segments), 256 threads per CTA:
//  - CTA (i, b, s) checks that row i sees every prefix row of its segment
//    (16-byte loads, 4 in flight per thread, byte loads for the unaligned
//    head and tail); segment 0 also gathers the row's T tree bytes into a
//    64-bit set with ballots.  S is chosen on the host so that the grid
//    covers every SM several times (the prefix lengths live on the device);
//  - a per-request ticket elects the last CTA, whose first warp derives each
//    parent (the highest visible node below i), checks the tree-mask rules
//    and writes the parent array and the ancestor bits.
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool all_ones(uint4 v) {
  // every byte nonzero
  auto ok = [](uint32_t w) { return ((w - 0x01010101u) & ~w & 0x80808080u) == 0; };
  return ok(v.x) && ok(v.y) && ok(v.z) && ok(v.w);
}

__global__ void __launch_bounds__(kThreads) mask_kernel(const MaskArgs a) {
  const int i = blockIdx.x, b = blockIdx.y, seg = blockIdx.z, nseg = gridDim.z, T = a.n_nodes;
  const int tid = threadIdx.x;
  const int64_t P = __ldg(a.prefix_lens + b);
  const int64_t start = __ldg(a.indptr + b), span = __ldg(a.indptr + b + 1) - start;
  const bool shape_ok = P >= 0 && span == (int64_t)T * (P + T);
  __shared__ int bad_prefix;
  __shared__ uint32_t half[2];
  __shared__ bool last;
  if (tid == 0) bad_prefix = 0;
  __syncthreads();
  uint64_t bits = 0;
  if (shape_ok) {
    const uint8_t* row = a.mask + start + (int64_t)i * (P + T);
    // This segment's prefix columns [c0, c1): all must be nonzero.
    const int64_t per = (P + nseg - 1) / nseg;
    const int64_t c0 = min((int64_t)seg * per, P), c1 = min(c0 + per, P);
    const uint8_t* part = row + c0;
    const int64_t len = c1 - c0;
    const int64_t align_gap = (int64_t)((16 - ((uintptr_t)part & 15)) & 15);
    const int64_t head = len < align_gap ? len : align_gap;
    bool ok = true;
    for (int64_t k = tid; k < head; k += kThreads) ok &= part[k] != 0;
    const int64_t nvec = (len - head) >> 4;
    const uint4* rv = reinterpret_cast<const uint4*>(part + head);
    for (int64_t k0 = tid; k0 < nvec; k0 += 4 * kThreads) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = k0 + u * kThreads;
        v[u] = k < nvec ? __ldg(rv + k) : make_uint4(~0u, ~0u, ~0u, ~0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) ok &= all_ones(v[u]);
    }
    for (int64_t k = head + 16 * nvec + tid; k < len; k += kThreads) ok &= part[k] != 0;
    if (!ok) atomicOr(&bad_prefix, 1);
    // Tree columns: bit j = row[P + j] != 0 (warps 0 and 1 cover j < 64).
    if (seg == 0 && tid < 64) {
      const uint32_t m = __ballot_sync(0xffffffffu, tid < T && row[P + tid] != 0);
      if ((tid & 31) == 0) half[tid >> 5] = m;
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (seg == 0) {
      if (shape_ok) bits = (uint64_t)half[0] | ((uint64_t)(T > 32 ? half[1] : 0u) << 32);
      a.rows[(size_t)b * T + i] = bits;
    }
    if (bad_prefix) atomicOr(a.status, DDTREE_ST_BAD_MASK);
    if (!shape_ok && i == 0 && seg == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
    __threadfence();
    last = atomicAdd(a.tickets + b, 1u) == (uint32_t)(T * nseg) - 1;
    if (last) __threadfence();
  }
  __syncthreads();
  if (!last || tid >= 32) return;
  // The request's rows are all in place: derive and check the tree.
  const int lane = tid;
  bool bad = false;
  for (int n = lane; n < T; n += 32) {
    const uint64_t r = __ldcg(reinterpret_cast<const unsigned long long*>(a.rows) + (size_t)b * T + n);
    const uint64_t below = r & ((n == 0) ? 0ull : (~0ull >> (64 - n)));
    const int p = below ? 63 - __clzll((long long)below) : -1;
    uint64_t want = 1ull << n;
    if (p >= 0) want |= __ldcg(reinterpret_cast<const unsigned long long*>(a.rows) + (size_t)b * T + p);
    if (shape_ok) bad |= r != want;
    a.parent[(size_t)b * T + n] = shape_ok ? p : -1;
    if (a.anc) a.anc[(size_t)b * T + n] = r;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, DDTREE_ST_BAD_MASK);
}

}  // namespace

cudaError_t launch_mask(const MaskArgs& a, cudaStream_t stream) {
  const int rows = a.n_nodes * a.batch;
  const int segs = std::max(1, std::min(64, (4 * a.num_sms + rows - 1) / rows));
  mask_kernel<<<dim3(a.n_nodes, a.batch, segs), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ddtree
