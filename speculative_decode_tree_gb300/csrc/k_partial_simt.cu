// Split-KV partial stage on CUDA cores (fp32 FMA).  The small-shape path and
// the correctness baseline of the tensor-core kernel.
//
// One CTA = one work item: 32 query rows of one request x one chunk of that
// request's key sequence ("Chunk 66.0": KV-split flash decode, partial +
// reduce).  Per tile of 32 keys it gathers the key rows through the
// page_size=1 index table with 16-byte loads ("Chunk 66.1": 128-bit bf16 KV
// loads), forms scores, applies the ancestor mask on tree keys only, runs an
// online softmax and accumulates O in registers.  It writes the chunk's
// normalised O_s and lse_s; the combine stage merges chunks.
#include "common.cuh"

namespace ddtree {
namespace {

constexpr int SR = 32;            // query rows per CTA
constexpr int SK = 32;            // keys per tile
constexpr int SROW = kRow + 8;    // padded smem row (bf16): 1168 B, 4-bank skew
constexpr int SPROW = SK + 1;     // padded score row (fp32)
constexpr int kThreads = 256;

constexpr size_t kSmemBytes = (size_t)(SR + SK) * SROW * 2 + (size_t)SR * SPROW * 4 +
                              SR * 4 * 3 + 64 * 8 + SK * 4;

__global__ void __launch_bounds__(kThreads) partial_simt_kernel(const VerifyArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem);
  uint16_t* sK = sQ + SR * SROW;
  float* sP = reinterpret_cast<float*>(sK + SK * SROW);
  float* sAlpha = sP + SR * SPROW;
  float* sM = sAlpha + SR;
  float* sL = sM + SR;
  uint64_t* sAnc = reinterpret_cast<uint64_t*>(sL + SR);
  int32_t* sIdx = reinterpret_cast<int32_t*>(sAnc + 64);

  const int tid = threadIdx.x;
  SplitLoc loc;
  if (!locate_split(a, blockIdx.y, loc)) return;
  const int row0 = blockIdx.x * SR;
  if (row0 >= a.rows_per_req) return;
  const int T = a.n_nodes, H = a.n_heads;
  const int slot = blockIdx.y;

  if (tid < T) sAnc[tid] = ancestor_bits(a.tree_parent + (size_t)loc.b * T, tid, T, a.status);

  // Q rows of this tile (rows past the request are zero).
  for (int e = tid; e < SR * (kRow / 8); e += kThreads) {
    int r = e / (kRow / 8), c = e % (kRow / 8);
    int row = row0 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < a.rows_per_req) {
      size_t g = (size_t)loc.b * a.rows_per_req + row;
      if (c < kLatent / 8)
        v = __ldg(reinterpret_cast<const uint4*>(a.q_latent + g * a.q_lat_stride) + c);
      else
        v = __ldg(reinterpret_cast<const uint4*>(a.q_rope + g * a.q_rope_stride) + (c - kLatent / 8));
    }
    *reinterpret_cast<uint4*>(sQ + r * SROW + c * 8) = v;
  }

  const int k_begin = loc.s * a.chunk_keys;
  const int k_end = min(k_begin + a.chunk_keys, loc.nkeys);

  float acc[SR][2];
#pragma unroll
  for (int r = 0; r < SR; ++r) acc[r][0] = acc[r][1] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // held by warp 0, lane = row

  const int sr = tid >> 3;   // score row
  const int sk = tid & 7;    // score key phase
  const int d0 = tid * 2;    // output dims owned by this thread

  for (int kt = k_begin; kt < k_end; kt += SK) {
    __syncthreads();  // previous tile fully consumed
    if (tid < SK) {
      int kp = kt + tid;
      int idx = -1;
      if (kp < k_end) {
        idx = __ldg(a.kv_indices + loc.idx_base + kp);
        if (idx < 0 || (a.pool_rows > 0 && idx >= a.pool_rows)) {
          atomicOr(a.status, DDTREE_ST_BAD_INDEX);
          idx = -1;
        }
      }
      sIdx[tid] = idx;
    }
    __syncthreads();
    for (int e = tid; e < SK * (kRow / 8); e += kThreads) {
      int k = e / (kRow / 8), c = e % (kRow / 8);
      int idx = sIdx[k];
      uint4 v = make_uint4(0, 0, 0, 0);
      if (idx >= 0) v = __ldg(reinterpret_cast<const uint4*>(a.kv_pool + (size_t)idx * kRow) + c);
      *reinterpret_cast<uint4*>(sK + k * SROW + c * 8) = v;
    }
    __syncthreads();

    // Scores: thread (sr, sk) does keys sk, sk+8, sk+16, sk+24 of row sr.
    {
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      const uint16_t* q = sQ + sr * SROW;
      for (int c = 0; c < kRow; c += 8) {
        uint4 qv = *reinterpret_cast<const uint4*>(q + c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 kv = *reinterpret_cast<const uint4*>(sK + (sk + 8 * j) * SROW + c);
          s[j] = fmaf(bf16_lo(qv.x), bf16_lo(kv.x), s[j]);
          s[j] = fmaf(bf16_hi(qv.x), bf16_hi(kv.x), s[j]);
          s[j] = fmaf(bf16_lo(qv.y), bf16_lo(kv.y), s[j]);
          s[j] = fmaf(bf16_hi(qv.y), bf16_hi(kv.y), s[j]);
          s[j] = fmaf(bf16_lo(qv.z), bf16_lo(kv.z), s[j]);
          s[j] = fmaf(bf16_hi(qv.z), bf16_hi(kv.z), s[j]);
          s[j] = fmaf(bf16_lo(qv.w), bf16_lo(kv.w), s[j]);
          s[j] = fmaf(bf16_hi(qv.w), bf16_hi(kv.w), s[j]);
        }
      }
      const int row = row0 + sr;
      const int node = row / H;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int k = sk + 8 * j;
        int kp = kt + k;
        bool ok = kp < k_end && sIdx[k] >= 0 && row < a.rows_per_req;
        if (ok && kp >= loc.P) ok = (sAnc[node] >> (kp - loc.P)) & 1ull;
        sP[sr * SPROW + k] = ok ? s[j] * a.sm_scale : -INFINITY;
      }
    }
    __syncthreads();

    // Online softmax: warp 0, one lane per row.
    if (tid < SR) {
      float* p = sP + tid * SPROW;
      float mx = -INFINITY;
      for (int k = 0; k < SK; ++k) mx = fmaxf(mx, p[k]);
      float m_new = fmaxf(m_run, mx);
      float alpha = 1.f, sum = 0.f;
      if (m_new != -INFINITY) {
        alpha = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
        for (int k = 0; k < SK; ++k) {
          float e = (p[k] == -INFINITY) ? 0.f : expf(p[k] - m_new);
          p[k] = e;
          sum += e;
        }
      } else {
        for (int k = 0; k < SK; ++k) p[k] = 0.f;
      }
      l_run = l_run * alpha + sum;
      m_run = m_new;
      sAlpha[tid] = alpha;
    }
    __syncthreads();

    // O[r, d0..d0+1] = alpha_r * O + sum_k p[r,k] V[k, d0..d0+1]
#pragma unroll
    for (int r = 0; r < SR; ++r) {
      float al = sAlpha[r];
      acc[r][0] *= al;
      acc[r][1] *= al;
    }
    for (int k = 0; k < SK; ++k) {
      uint32_t v = *reinterpret_cast<const uint32_t*>(sK + k * SROW + d0);
      float v0 = bf16_lo(v), v1 = bf16_hi(v);
#pragma unroll
      for (int r = 0; r < SR; ++r) {
        float p = sP[r * SPROW + k];
        acc[r][0] = fmaf(p, v0, acc[r][0]);
        acc[r][1] = fmaf(p, v1, acc[r][1]);
      }
    }
  }

  if (tid < SR) {
    sM[tid] = m_run;
    sL[tid] = l_run;
  }
  __syncthreads();
  uint16_t* po = a.partial_o + (size_t)slot * a.rows_per_req * kLatent;
  float* pl = a.partial_lse + (size_t)slot * a.rows_per_req;
#pragma unroll
  for (int r = 0; r < SR; ++r) {
    int row = row0 + r;
    if (row >= a.rows_per_req) break;
    float l = sL[r];
    float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<__nv_bfloat162*>(po + (size_t)row * kLatent + d0) =
        __floats2bfloat162_rn(acc[r][0] * inv, acc[r][1] * inv);
    if (tid == 0) pl[row] = l > 0.f ? sM[r] + logf(l) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_partial_simt(const VerifyArgs& a, cudaStream_t stream) {
  // The shared-memory opt-in is per device; set it once for each.
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(partial_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(a.row_tiles, a.total_splits);
  partial_simt_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ddtree
