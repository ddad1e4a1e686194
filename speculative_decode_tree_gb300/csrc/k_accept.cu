// Greedy acceptance of a verified draft tree, and the KV commit that follows
// ("Chunk 66.0": the DDTree commit length is the number of tokens one verify
// step commits).
//
// Stage 1 (argmax): the target's token at every scored position is the argmax
// of its logits row (first index among equal maxima).  A row of the vocabulary
// (129,280 bf16 for DeepSeek-V3, 253 KB) is split into segments so that the
// grid covers every SM several times; each CTA streams its segment with 16-byte
// loads, reduces (value, index) in registers, warp shuffles and shared memory,
// and folds the result into the row's 64-bit key with one atomicMax.  The key
// orders by value, then by smaller index: (order-preserving bits of the value
// << 32) | (0xffffffff - index).  The whole stage is one pass over the logits:
// HBM-bound.
//
// Stage 2 (walk + commit): one warp per request walks the tree from the prefix
// end.  At each step every lane tests two nodes (T <= 64) for "child of the
// current node and drafted the predicted token"; a ballot picks the smallest
// such node.  The warp then writes the accepted path, the next token, the pool
// rows of the accepted nodes in path order (committed context) and those of
// the other nodes in node order (released rows).
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int kArgmaxThreads = 256;

__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t idx) {
  if (v == 0.f) v = 0.f;  // -0 and +0 compare equal: one code for both
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xffffffffu - idx);
}

__device__ __forceinline__ void take(float v, uint32_t i, float& bv, uint32_t& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

// Row blockIdx.x of the logits, elements [seg*len, (seg+1)*len) with seg = blockIdx.y.
__device__ __forceinline__ void argmax_segment(const uint16_t* __restrict__ logits, int vocab, int seg_len,
                                               uint64_t* keys) {
  const int row = blockIdx.x;
  const int64_t begin = (int64_t)blockIdx.y * seg_len;
  const int64_t end = begin + seg_len < (int64_t)vocab ? begin + seg_len : (int64_t)vocab;
  const uint16_t* x = logits + (int64_t)row * vocab;
  float bv = -INFINITY;
  uint32_t bi = 0xffffffffu;
  // 16-byte loads where the row (and segment) start allows them.
  const bool vec = ((((uintptr_t)(x + begin)) & 15) == 0);
  int64_t i = begin;
  if (vec) {
    const int64_t nvec = (end - begin) >> 3;
    const uint4* xv = reinterpret_cast<const uint4*>(x + begin);
    // Four independent 16-byte loads in flight per thread and iteration.
    for (int64_t k0 = threadIdx.x; k0 < nvec; k0 += 4 * kArgmaxThreads) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = k0 + u * kArgmaxThreads;
        w[u] = k < nvec ? __ldg(xv + k) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t base = (uint32_t)(begin + 8 * (k0 + u * kArgmaxThreads));
        take(bf16_lo(w[u].x), base + 0, bv, bi);
        take(bf16_hi(w[u].x), base + 1, bv, bi);
        take(bf16_lo(w[u].y), base + 2, bv, bi);
        take(bf16_hi(w[u].y), base + 3, bv, bi);
        take(bf16_lo(w[u].z), base + 4, bv, bi);
        take(bf16_hi(w[u].z), base + 5, bv, bi);
        take(bf16_lo(w[u].w), base + 6, bv, bi);
        take(bf16_hi(w[u].w), base + 7, bv, bi);
      }
    }
    i = begin + 8 * nvec;
  }
  for (int64_t k = i + threadIdx.x; k < end; k += kArgmaxThreads)
    take(__uint_as_float((uint32_t)__ldg(x + k) << 16), (uint32_t)k, bv, bi);

  // Reduce the CTA's candidates as keys (order: value, then smaller index).
  uint64_t key = bi == 0xffffffffu ? 0ull : argmax_key(bv, bi);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other > key ? other : key;
  }
  __shared__ uint64_t red[kArgmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = key;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgmaxThreads / 32; ++w) key = red[w] > key ? red[w] : key;
    if (key) atomicMax(reinterpret_cast<unsigned long long*>(keys + row), (unsigned long long)key);
  }
}

struct WalkArgs {
  const int32_t* draft;
  const int32_t* parent;
  const int32_t* kv_indices;
  const int32_t* kv_indptr;
  const int32_t* prefix_lens;
  const uint64_t* keys;  // [B, T+1]
  uint32_t* tickets;     // [B]: CTAs of the request done with their argmax
  int32_t* accept_len;
  int32_t* next_token;
  int32_t* accepted_nodes;
  int32_t* commit_indices;
  int32_t* freed_indices;
  uint32_t* status;
  int n_nodes;
};

// The walk and commit of request b by one warp (lane = 0..31).  The argmax
// keys were written by other CTAs' atomics: read them through L2.
__device__ void walk_request(const WalkArgs& a, int b, int lane, int32_t* pred, int32_t* path, int32_t* rows) {
  const int T = a.n_nodes;
  // Every load the walk needs is issued up front (one memory round trip),
  // then the tree rows' pool indices (a second one, overlapping the walk).
  const int j0 = lane, j1 = lane + 32;
  const bool v0 = j0 < T, v1 = j1 < T;
  const int32_t* par = a.parent + (size_t)b * T;
  const int32_t* dr = a.draft + (size_t)b * T;
  const unsigned long long* keys = reinterpret_cast<const unsigned long long*>(a.keys) + (size_t)b * (T + 1);
  const uint64_t k0 = (lane <= T) ? __ldcg(keys + lane) : 0ull;
  const uint64_t k1 = (lane + 32 <= T) ? __ldcg(keys + lane + 32) : 0ull;
  const uint64_t k2 = (lane == 0 && T == 64) ? __ldcg(keys + 64) : 0ull;
  const int p0 = v0 ? __ldg(par + j0) : -2, p1 = v1 ? __ldg(par + j1) : -2;
  const int d0 = v0 ? __ldg(dr + j0) : 0, d1 = v1 ? __ldg(dr + j1) : 0;
  const int P = __ldg(a.prefix_lens + b);
  const int ip0 = __ldg(a.kv_indptr + b), ip1 = __ldg(a.kv_indptr + b + 1);
  const bool lengths_ok = P >= 0 && ip1 - ip0 == P + T;
  const int64_t base = (int64_t)ip0 + P;
  if (lengths_ok) {
    if (v0) rows[j0] = __ldg(a.kv_indices + base + j0);
    if (v1) rows[j1] = __ldg(a.kv_indices + base + j1);
  }
  auto tok = [](uint64_t k) { return (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffu)); };
  if (lane <= T) pred[lane] = tok(k0);
  if (lane + 32 <= T) pred[lane + 32] = tok(k1);
  if (lane == 0 && T == 64) pred[64] = tok(k2);
  if ((v0 && (p0 < -1 || p0 >= j0)) || (v1 && (p1 < -1 || p1 >= j1))) atomicOr(a.status, DDTREE_ST_BAD_PARENT);
  if (!lengths_ok && lane == 0) atomicOr(a.status, DDTREE_ST_BAD_LENGTH);
  __syncwarp();

  int cur = -1, y = pred[0], len = 0;
  uint64_t on_path = 0;
  for (int step = 0; step < T; ++step) {
    const uint32_t m0 = __ballot_sync(0xffffffffu, v0 && p0 == cur && d0 == y);
    const uint32_t m1 = __ballot_sync(0xffffffffu, v1 && p1 == cur && d1 == y);
    if (!(m0 | m1)) break;
    const int c = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
    if (c <= cur) break;  // a malformed tree cannot loop the walk
    if (lane == 0) path[len] = c;
    on_path |= 1ull << c;
    ++len;
    cur = c;
    y = pred[1 + c];
  }
  __syncwarp();

  if (lane == 0) {
    a.accept_len[b] = len;
    a.next_token[b] = y;
  }
  const size_t o = (size_t)b * T;
  const uint64_t all = T >= 64 ? ~0ull : ((1ull << T) - 1);
  const uint64_t off = all & ~on_path;
  for (int k = lane; k < T; k += 32) {
    const int node = k < len ? path[k] : -1;
    a.accepted_nodes[o + k] = node;
    a.commit_indices[o + k] = (node >= 0 && lengths_ok) ? rows[node] : -1;
    // The k-th node (in node order) that is not on the path.
    int freed = -1;
    if (k < T - len && lengths_ok) {
      uint64_t m = off;
      for (int s = 0; s < k; ++s) m &= m - 1;  // drop the k lowest set bits
      freed = rows[__ffsll((long long)m) - 1];
    }
    a.freed_indices[o + k] = freed;
  }
}


// grid = (rows, segments), rows = B (T+1) ordered request by request.  Each
// CTA folds its segment's argmax into the row key; the last CTA of a request
// to finish (a ticket per request) then walks that request's tree, so the
// whole step is one launch.
__global__ void __launch_bounds__(kArgmaxThreads) accept_kernel(const uint16_t* __restrict__ logits, int vocab,
                                                                int seg_len, const WalkArgs a) {
  __shared__ int32_t pred[DDTREE_MAX_NODES + 1];
  __shared__ int32_t path[DDTREE_MAX_NODES];
  __shared__ int32_t rows[DDTREE_MAX_NODES];
  __shared__ bool last;
  argmax_segment(logits, vocab, seg_len, const_cast<uint64_t*>(a.keys));
  const int T1 = a.n_nodes + 1;
  const int b = blockIdx.x / T1;
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's key update before its ticket
    const uint32_t done = atomicAdd(a.tickets + b, 1u);
    last = done == (uint32_t)(T1 * gridDim.y) - 1;
    if (last) __threadfence();  // every other CTA's key update before the walk reads
  }
  __syncthreads();
  if (last && threadIdx.x < 32) walk_request(a, b, threadIdx.x, pred, path, rows);
}
}  // namespace

cudaError_t launch_accept(const AcceptArgs& x, cudaStream_t stream) {
  const int rows = x.batch * (x.n_nodes + 1);
  // Enough CTAs to cover the SMs about four times; each reads >= 4096 logits.
  int segs = (4 * x.num_sms + rows - 1) / rows;
  const int max_segs = (x.vocab + 4095) / 4096;
  segs = max(1, min(segs, max_segs));
  int seg_len = (x.vocab + segs - 1) / segs;
  seg_len = (seg_len + 7) & ~7;  // keeps segment starts 16-byte aligned when rows are
  segs = (x.vocab + seg_len - 1) / seg_len;
  WalkArgs w;
  w.draft = x.draft;
  w.parent = x.parent;
  w.kv_indices = x.kv_indices;
  w.kv_indptr = x.kv_indptr;
  w.prefix_lens = x.prefix_lens;
  w.keys = x.keys;
  w.tickets = x.tickets;
  w.accept_len = x.accept_len;
  w.next_token = x.next_token;
  w.accepted_nodes = x.accepted_nodes;
  w.commit_indices = x.commit_indices;
  w.freed_indices = x.freed_indices;
  w.status = x.status;
  w.n_nodes = x.n_nodes;
  accept_kernel<<<dim3(rows, segs), kArgmaxThreads, 0, stream>>>(x.logits, x.vocab, seg_len, w);
  return cudaGetLastError();
}

}  // namespace ddtree
