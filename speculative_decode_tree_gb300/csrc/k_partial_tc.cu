// Split-KV partial stage on the tcgen05 tensor cores (sm_103a).
//
// One work item = 128 query rows (node-major (node, head) rows of one request)
// x one chunk of that request's key sequence, run by a cluster of two CTAs
// with different jobs ("Chunk 66.0": KV-split flash decode, partial + reduce;
// the split count is the plan's, "Chunk 66.1"):
//
//  scorer (cluster rank 0)
//    Q latent (128 x 512 bf16) lives in TMEM as the A operand, Q rope in
//    shared memory; per tile of 128 keys it gathers the 576-wide key rows
//    through the page_size=1 index table with TMA row gathers (4 rows per
//    instruction, "Chunk 66.1": wide KV loads) into 128-byte-swizzled chunks
//    of 64 columns, or with one 2-D TMA tile load per chunk when the tile's
//    128 indices are one contiguous run (defragmented KV),
//    issues S = Q K^T (M=128, N=128, K=576) into one of two TMEM S buffers,
//    and four softmax warps (one query row per thread) apply the ancestor
//    mask on tree keys only, keep a running max with lazy rescaling, and
//    write P = exp(s - m) as a bf16 K-major tile plus per-row rescale
//    factors, which one thread ships to the peer with a bulk shared-memory
//    copy across the cluster.
//  accumulator (cluster rank 1)
//    holds O (128 x 512 fp32) in all 512 TMEM columns, gathers the value
//    rows (first 512 columns of the same keys) as MN-major operands, and
//    issues O += P V (M=128, N=128 per quarter, K=128 keys) from the P tiles
//    it receives.  Its epilogue warps rescale O rows when the scorer's
//    running max moved (rare), and at the end write O_s = O / l.
//
// Work per (row, key): 576 MACs on the scorer, 512 on the accumulator.
// Every mbarrier wait is bounded; on expiry the kernel sets
// DDTREE_ST_TIMEOUT, stops issuing work, waits (bounded) for its own
// tensor-core work and frees its TMEM.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace ddtree {
namespace {

using namespace ptx;

constexpr int TK = 128;                 // keys per tile
constexpr int ROWS = 128;               // query rows per work item
constexpr int CHUNK = 16384;            // one 64-column chunk of a tile: 128 keys x 128 B
constexpr int QRING = 10;               // scorer key-chunk slots
constexpr int VRING = 4;                // accumulator slots, each a pair of chunks (32 KB)
constexpr int PTILE = 32768;            // bf16 P tile: 2 swizzle atoms of 128 rows x 128 B
constexpr int META = 1040;              // alpha[128], lfin[128], flag words[4]
constexpr int PCOPY = PTILE + META;     // bytes shipped per tile (multiple of 16)
constexpr int PBUF = 34816;             // P buffer stride (1024-aligned)
constexpr int kThreads = 384;                  // 12 warps
constexpr float kLazyRescale = 8.0f;    // rescale only when the max grows by > 2^8 (log2 units)
constexpr uint64_t kWaitNs = 2000000000ull;

// Shared-memory map (offsets from a 1024-aligned base).
constexpr int Q_ROPE = 0;                               // scorer: 16 KB
constexpr int Q_RING = Q_ROPE + CHUNK;                  // scorer: 8 x 16 KB
constexpr int Q_STAGE = Q_RING + QRING * CHUNK;         // scorer: 1 x PBUF (P staging)
constexpr int Q_END = Q_STAGE + PBUF;
constexpr int V_PBUF = 0;                               // accumulator: 2 x PBUF
constexpr int V_RING = V_PBUF + 2 * PBUF;               // accumulator: 4 x 32 KB
constexpr int V_END = V_RING + VRING * 2 * CHUNK;
constexpr int BIG_END = (Q_END > V_END ? Q_END : V_END);

struct __align__(8) Ctrl {
  uint64_t kfull[QRING], kempty[QRING];  // scorer ring (QRING <= 16)
  uint64_t sfull[2], sempty[2];          // scorer S buffers
  uint64_t pfree[2];                     // scorer: peer released P buffer (2 arrivals)
  uint64_t vfull[VRING], vempty[VRING];  // accumulator ring
  uint64_t pfull[2];                     // accumulator: P tile landed (tx)
  uint64_t pvdone[2];                    // accumulator: PV of a tile finished
  uint64_t corr_done;                    // accumulator: O rows rescaled
  uint64_t mma_done;                     // last tensor-core work of this CTA finished
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t key_mask[2][4];               // scorer: valid-key bits per tile parity
  uint32_t pad_;
  uint64_t anc[64];
  int32_t par[64];   // the request's parents, staged for the ancestor walk                      // scorer: ancestor bits per node
};

constexpr size_t kSmemBytes = 1024 + BIG_END + sizeof(Ctrl) + 64;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ void set_abort(Ctrl* c, uint32_t* status) {
  c->abort = 1;
  atomicOr(status, DDTREE_ST_TIMEOUT);
}

// Bounded wait; on expiry mark the CTA aborted.  Returns false when aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctrl* c, uint32_t* status) {
  if (*(volatile uint32_t*)&c->abort) return false;
  if (mbar_wait(bar, parity, kWaitNs)) return true;
  set_abort(c, status);
  return false;
}
__device__ __forceinline__ bool wait_cluster_or_abort(uint64_t* bar, uint32_t parity, Ctrl* c,
                                                      uint32_t* status) {
  if (*(volatile uint32_t*)&c->abort) return false;
  if (mbar_wait_cluster(bar, parity, kWaitNs)) return true;
  set_abort(c, status);
  return false;
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads,
// so every thread takes the same decision (used to stop after an abort).
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0;\n"
      "  bar.red.or.pred q, %2, %3, p;\n"
      "  selp.u32 %0, 1, 0, q; }"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ bool aborted(Ctrl* c) { return *(volatile uint32_t*)&c->abort != 0; }

struct Item {
  SplitLoc loc;
  int row0;      // first query row of the tile within the request
  int k_begin;   // first key of the chunk
  int k_end;     // one past the last key
  int ntiles;
  int slot;      // split slot in the workspace
};

// TMA maps of the KV pool: rows of 576 bf16, 128-byte swizzle; `row4` has a
// one-row box for tile::gather4, `tile` a 128-row box for contiguous runs.
struct PoolMaps {
  CUtensorMap row4;
  CUtensorMap tile;
};

// One tile's 128 key indices as this lane sees them: keys 4*lane .. 4*lane+3
// (out-of-range and past-the-chunk keys become -1, which TMA fills with
// zeros), plus whether the whole tile is one contiguous, fully valid run.
struct TileIdx {
  int4 k4;
  int first;
  bool contiguous;
};

// Raw index loads of one tile for this lane (no use of the values, so the
// loads can be issued a tile early); finish_tile_indices validates them.
struct RawIdx {
  int v[4];
};
__device__ __forceinline__ RawIdx raw_tile_indices(const VerifyArgs& a, const Item& it, int tile, int lane) {
  const int k0 = it.k_begin + tile * TK + 4 * lane;
  RawIdx r;
#pragma unroll
  for (int j = 0; j < 4; ++j) r.v[j] = (k0 + j < it.k_end) ? __ldg(a.kv_indices + it.loc.idx_base + k0 + j) : -1;
  return r;
}
__device__ __forceinline__ TileIdx finish_tile_indices(const VerifyArgs& a, RawIdx r, int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (r.v[j] < 0 || (a.pool_rows > 0 && r.v[j] >= a.pool_rows)) r.v[j] = -1;
  TileIdx t;
  t.k4 = make_int4(r.v[0], r.v[1], r.v[2], r.v[3]);
  t.first = __shfl_sync(0xffffffffu, r.v[0], 0);
  const bool run = r.v[0] >= 0 && r.v[0] == t.first + 4 * lane && r.v[1] == r.v[0] + 1 &&
                   r.v[2] == r.v[0] + 2 && r.v[3] == r.v[0] + 3;
  t.contiguous = __all_sync(0xffffffffu, run);
  return t;
}

// Producer warps.  Scorer: warps 0, 2, 3, 8..11 (7); accumulator: warps 0, 3,
// 8..11 (6).  Returns the producer rank of `warp`, or -1.
constexpr int kScorerProducers = 7;
constexpr int kAccProducers = 6;
__device__ __forceinline__ int producer_rank(int warp, bool scorer) {
  if (warp == 0) return 0;
  if (scorer && warp == 2) return 1;
  if (warp == 3) return scorer ? 2 : 1;
  if (warp >= 8) return warp - (scorer ? 5 : 6);
  return -1;
}

// The key indices this producer lane copies for its four-key groups
// g = rank, rank + np, ... (lane covers key 4g + lane/8, 16-byte piece lane%8).
struct MyKeys {
  int id[6];  // ceil(32 / producers) groups at most
  int n;
};
__device__ __forceinline__ MyKeys my_keys(const TileIdx& ti, int lane, int rank, int np) {
  MyKeys mk;
  mk.n = 0;
  const int sel = lane >> 3;
#pragma unroll
  for (int j = 0; j < 6; ++j) {
    const int g = rank + j * np;
    const int x = __shfl_sync(0xffffffffu, ti.k4.x, g & 31);
    const int y = __shfl_sync(0xffffffffu, ti.k4.y, g & 31);
    const int z = __shfl_sync(0xffffffffu, ti.k4.z, g & 31);
    const int w = __shfl_sync(0xffffffffu, ti.k4.w, g & 31);
    mk.id[j] = sel == 0 ? x : sel == 1 ? y : sel == 2 ? z : w;
    if (g < 32) mk.n = j + 1;
  }
  return mk;
}

// Fills `nchunks` 64-column chunks (columns 64*c0 ...) of the tile into
// `dst` (chunk stride CHUNK; row k at +128 k, 128-byte swizzled) and arrives
// on `bar` once per lane.  Scattered tiles: 16-byte cp.async of this warp's
// key groups (zero-filled for invalid keys).  Contiguous tiles: rank 0 adds
// the bytes to `bar` and loads each chunk with one 2-D TMA tile; the others
// only arrive.  `bar` expects 32 arrivals per producer warp.
__device__ __forceinline__ void fill_chunks(const PoolMaps& maps, const uint16_t* pool, uint8_t* dst, int c0,
                                            int nchunks, const TileIdx& ti, const MyKeys& mk, int rank, int np,
                                            int lane, uint64_t* bar) {
  if (ti.contiguous) {
    if (rank == 0 && lane == 0) {
      mbar_expect_tx(bar, nchunks * CHUNK);
      for (int c = 0; c < nchunks; ++c)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(smem_u32(dst + c * CHUNK)), "l"(&maps.tile), "r"((c0 + c) * 64), "r"(ti.first),
              "r"(smem_u32(bar))
            : "memory");
    }
    __syncwarp();
  } else {
    const int piece = lane & 7;
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t base = smem_u32(dst + c * CHUNK);
#pragma unroll
      for (int j = 0; j < 6; ++j) {
        if (j < mk.n) {
          const int key = 4 * (rank + j * np) + (lane >> 3);
          const int id = mk.id[j];
          const uint16_t* src = pool + (size_t)(id < 0 ? 0 : id) * kRow + (c0 + c) * 64 + piece * 8;
          cp_async16_zfill(base + key * 128 + ((piece ^ (key & 7)) << 4), src, id < 0 ? 0u : 16u);
        }
      }
    }
  }
  cp_async_mbar_arrive(bar);
}

// Pulls the whole 1152-byte rows of one tile's keys into L2 with one bulk
// prefetch per row (through this SM's otherwise idle TMA unit); thread r of
// 128 handles key r.  Issued by the accumulator a few tiles ahead
// of the scorer, so the scorer's gathers hit L2 instead of waiting on DRAM.
constexpr int kL2Ahead = 3;
__device__ __forceinline__ void prefetch_tile_l2(const VerifyArgs& a, const Item& it, int tile, int r) {
  if (tile >= it.ntiles) return;
  const int kp = it.k_begin + tile * TK + r;
  if (kp >= it.k_end) return;
  const int id = __ldg(a.kv_indices + it.loc.idx_base + kp);
  if (id < 0 || (a.pool_rows > 0 && id >= a.pool_rows)) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.kv_pool + (size_t)id * kRow), "r"(kRow * 2)
               : "memory");
}

// ------------------------------------------------------------------ scorer
__device__ void scorer(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;        // cols [0,256): Q latent; [256,384), [384,512): S
  const uint32_t peer = 1;

  const int prank = producer_rank(warp, true);
  if (prank >= 0) {
    // ---- producers: key chunks 0..8 of every tile
    int n = 0;
    // Indices are loaded one tile ahead so their latency hides behind a
    // tile's worth of copies.
    RawIdx raw_next = raw_tile_indices(a, it, 0, lane);
    for (int t = 0; t < it.ntiles; ++t) {
      const TileIdx ti = finish_tile_indices(a, raw_next, lane);
      if (t + 1 < it.ntiles) raw_next = raw_tile_indices(a, it, t + 1, lane);
      const MyKeys mk = my_keys(ti, lane, prank, kScorerProducers);
      for (int ch = 0; ch < 9; ++ch, ++n) {
        const int slot = n % QRING;
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&c->kempty[slot], ((n / QRING) & 1) ^ 1, c, a.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          return;
        }
        fill_chunks(maps, a.kv_pool, sm + Q_RING + slot * CHUNK, ch, 1, ti, mk, prank, kScorerProducers, lane,
                    &c->kfull[slot]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1) {
    // ---- MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      const uint64_t rope_desc = desc_sw128(smem_u32(sm + Q_ROPE), 16, 1024);
      int n = 0;
      bool ok = true;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int s = t & 1;
        const uint32_t sbuf = tmem + 256 + 128 * s;
        if (!wait_or_abort(&c->sempty[s], ((t >> 1) & 1) ^ 1, c, a.status)) { ok = false; break; }
        tc_fence_after();
        for (int ch = 0; ch < 9; ++ch, ++n) {
          const int slot = n % QRING;
          if (!wait_or_abort(&c->kfull[slot], (n / QRING) & 1, c, a.status)) { ok = false; break; }
          fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
          const uint64_t kdesc = desc_sw128(smem_u32(sm + Q_RING + slot * CHUNK), 16, 1024);
          if (ch < 8) mma_ts_x4(sbuf, tmem + ch * 32, kdesc, idesc, ch > 0);  // latent: Q from TMEM
          else mma_ss_x4<2, 2>(sbuf, rope_desc, kdesc, idesc, 1);            // rope: Q from shared memory
          mma_commit(&c->kempty[slot]);
        }
        if (ok) mma_commit(&c->sfull[s]);
      }
      mma_commit(&c->mma_done);
    }
  } else if (warp >= 4) {
    // ---- softmax: thread = query row r
    const int r = tid - 128;
    const int w = warp - 4;
    const int req_row = it.row0 + r;
    const bool row_ok = req_row < a.rows_per_req;
    const uint64_t anc = row_ok ? c->anc[req_row / a.n_heads] : 0ull;
    const float scale2 = a.sm_scale * 1.4426950408889634f;  // scores in log2 units
    float m_ref = -INFINITY, l = 0.f;
    const uint32_t my_lane_addr = (uint32_t)(w * 32) << 16;
    const uint32_t peer_pbuf = map_cluster(smem_u32(sm + V_PBUF), peer);
    const uint32_t peer_pfull = map_cluster(smem_u32(&c->pfull[0]), peer);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      const int k0 = it.k_begin + t * TK;
      // Valid-key bits of this tile: warp w covers keys 32w .. 32w+31.
      {
        const int kp = k0 + 32 * w + lane;
        bool v = false;
        if (kp < it.k_end) {
          const int id = __ldg(a.kv_indices + it.loc.idx_base + kp);
          v = id >= 0 && (a.pool_rows <= 0 || id < a.pool_rows);
          if (!v) atomicOr(a.status, DDTREE_ST_BAD_INDEX);
        }
        const uint32_t bits = __ballot_sync(0xffffffffu, v);
        if (lane == 0) c->key_mask[s][w] = bits;
      }
      wait_or_abort(&c->sfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      tc_fence_after();
      uint32_t xr[4][32];  // raw fp32 scores of this row, 128 keys
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tmem + my_lane_addr + 256 + 128 * s + 32 * q, xr[q]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->sempty[s]);
      named_bar(1, 128);  // key_mask of this tile visible; previous tile's staging reads done
      uint32_t km[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) km[q] = c->key_mask[s][q];
      // Tiles of valid prefix keys only (the common case) need no mask.
      const bool plain = (k0 + TK <= it.loc.P) && (k0 + TK <= it.k_end) &&
                         ((km[0] & km[1] & km[2] & km[3]) == 0xffffffffu);
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (plain && row_ok) {
#pragma unroll
        for (int k = 0; k < TK; ++k) mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(xr[k >> 5][k & 31]));
      } else {
#pragma unroll
        for (int k = 0; k < TK; ++k) {
          const int kp = k0 + k;
          bool ok = row_ok && ((km[k >> 5] >> (k & 31)) & 1u);
          if (ok && kp >= it.loc.P) ok = (anc >> (kp - it.loc.P)) & 1ull;
          const float v = ok ? __uint_as_float(xr[k >> 5][k & 31]) : -INFINITY;
          xr[k >> 5][k & 31] = __float_as_uint(v);
          mx[k & 3] = fmaxf(mx[k & 3], v);
        }
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale2;
      float alpha = 1.f;
      if (mt > m_ref + kLazyRescale) {  // also true on the first finite max
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
        m_ref = mt;
      }
      const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // The staging buffer is free once the previous tile's copy has read it
      // (long done by now: a whole QK^T tile passed since it was issued).
      if (r == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      named_bar(1, 128);
      uint8_t* stg = sm + Q_STAGE;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {  // 16-byte chunk cc = keys 8cc .. 8cc+7
        uint32_t pk[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int k = 8 * cc + 2 * h;
          const float p0 = ex2_approx(fmaf(__uint_as_float(xr[k >> 5][k & 31]), scale2, nm));
          const float p1 = ex2_approx(fmaf(__uint_as_float(xr[(k + 1) >> 5][(k + 1) & 31]), scale2, nm));
          ps[h] += p0 + p1;
          __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
          pk[h] = *reinterpret_cast<uint32_t*>(&b);
        }
        const int atom = cc >> 3, c16 = cc & 7;
        *reinterpret_cast<uint4*>(stg + atom * CHUNK + r * 128 + ((c16 ^ (r & 7)) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      const float sum = (row_ok ? 1.f : 0.f) * ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      l = l * alpha + sum;
      float* meta = reinterpret_cast<float*>(stg + PTILE);
      meta[r] = alpha;
      meta[128 + r] = l;
      const uint32_t flag = __ballot_sync(0xffffffffu, t > 0 && alpha != 1.f);
      if (lane == 0) reinterpret_cast<uint32_t*>(meta + 256)[w] = flag;
      fence_async_smem();
      named_bar(1, 128);
      if (r == 0 && !aborted(c)) {
        // The peer's P buffer s is free once it finished tile t-2.
        if (wait_cluster_or_abort(&c->pfree[s], ((t >> 1) & 1) ^ 1, c, a.status)) {
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
              "cp.async.bulk.commit_group;" ::"r"(peer_pbuf + s * PBUF),
              "r"(smem_u32(stg)), "r"(PCOPY), "r"(peer_pfull + s * 8)
              : "memory");
        }
      }
      if (named_bar_or(1, 128, aborted(c))) break;
    }
    if (row_ok) {
      a.partial_lse[(size_t)it.slot * a.rows_per_req + req_row] =
          (l > 0.f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    if (r == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

// ------------------------------------------------------------ accumulator
__device__ void accumulator(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;  // O: cols [0,512)
  const uint32_t peer = 0;

  const int prank = producer_rank(warp, false);
  if (prank >= 0) {
    // ---- producers: value chunk pairs (0,1) .. (6,7) of every tile
    int n = 0;
    RawIdx raw_next = raw_tile_indices(a, it, 0, lane);
    for (int t = 0; t < it.ntiles; ++t) {
      const TileIdx ti = finish_tile_indices(a, raw_next, lane);
      if (t + 1 < it.ntiles) raw_next = raw_tile_indices(a, it, t + 1, lane);
      const MyKeys mk = my_keys(ti, lane, prank, kAccProducers);
      for (int q = 0; q < 4; ++q, ++n) {
        const int slot = n % VRING;
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&c->vempty[slot], ((n / VRING) & 1) ^ 1, c, a.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          return;
        }
        fill_chunks(maps, a.kv_pool, sm + V_RING + slot * 2 * CHUNK, 2 * q, 2, ti, mk, prank, kAccProducers, lane,
                    &c->vfull[slot]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);  // A = P K-major, B = V MN-major
      for (int s = 0; s < 2; ++s) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
      int n = 0;
      uint32_t corr_ph = 0;
      bool ok = true;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int s = t & 1;
        if (!wait_or_abort(&c->pfull[s], (t >> 1) & 1, c, a.status)) { ok = false; break; }
        const uint32_t* flags = reinterpret_cast<const uint32_t*>(sm + V_PBUF + s * PBUF + PTILE + 1024);
        if (flags[0] | flags[1] | flags[2] | flags[3]) {
          if (!wait_or_abort(&c->corr_done, corr_ph, c, a.status)) { ok = false; break; }
          corr_ph ^= 1;
        }
        tc_fence_after();
        const uint64_t pdesc = desc_sw128(smem_u32(sm + V_PBUF + s * PBUF), 16, 1024);
        for (int q = 0; q < 4; ++q, ++n) {
          const int slot = n % VRING;
          if (!wait_or_abort(&c->vfull[slot], (n / VRING) & 1, c, a.status)) { ok = false; break; }
          fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
          const uint64_t vdesc = desc_sw128(smem_u32(sm + V_RING + slot * 2 * CHUNK), CHUNK, 1024);
          // K steps 0..3 read P atom 0 (keys 0..63), 4..7 atom 1; V advances
          // 16 keys (2 KB) per step.
          mma_ss_x4<2, 128>(tmem + 128 * q, pdesc, vdesc, idesc, t > 0 ? 1u : 0u);
          mma_ss_x4<2, 128>(tmem + 128 * q, pdesc + (CHUNK >> 4), vdesc + 512, idesc, 1u);
          mma_commit(&c->vempty[slot]);
        }
        if (ok) mma_commit(&c->pvdone[s]);
      }
      mma_commit(&c->mma_done);
    }
  } else if (warp == 2) {
    // ---- relay: when PV of tile t finished, re-arm the P buffer and tell
    // the scorer (first of its two releases of that buffer).
    if (lane == 0) {
      const uint32_t peer_pfree = map_cluster(smem_u32(&c->pfree[0]), peer);
      for (int t = 0; t < it.ntiles; ++t) {
        const int s = t & 1;
        if (!wait_or_abort(&c->pvdone[s], (t >> 1) & 1, c, a.status)) break;
        if (t + 2 < it.ntiles) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(peer_pfree + s * 8)
                     : "memory");
      }
    }
  } else if (warp >= 4) {
    // ---- correction + epilogue: thread = row r (TMEM lane r)
    const int r = tid - 128;
    const int w = warp - 4;
    const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
    const uint32_t peer_pfree = map_cluster(smem_u32(&c->pfree[0]), peer);
    float lfin = 0.f;
    for (int t = 0; t < kL2Ahead; ++t) prefetch_tile_l2(a, it, t, r);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      prefetch_tile_l2(a, it, t + kL2Ahead, r);
      wait_or_abort(&c->pfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      const uint8_t* pb = sm + V_PBUF + s * PBUF;
      const float* meta = reinterpret_cast<const float*>(pb + PTILE);
      const uint32_t* flags = reinterpret_cast<const uint32_t*>(meta + 256);
      lfin = meta[128 + r];
      if (flags[0] | flags[1] | flags[2] | flags[3]) {
        const float alpha = meta[r];
        // O must hold PV of tiles < t before it is rescaled.
        wait_or_abort(&c->pvdone[(t - 1) & 1], ((t - 1) >> 1) & 1, c, a.status);
        tc_fence_after();
        // tcgen05.ld/st are warp-collective: the whole warp takes part when
        // any of its rows needs rescaling (alpha == 1 leaves a row unchanged).
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t v[16];
          for (int q = 0; q < 32; ++q) {
            tmem_ld16(lane_addr + 16 * q, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(lane_addr + 16 * q, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->corr_done);
      }
      // Second release of P buffer s: its metadata has been read.
      const bool stop = named_bar_or(2, 128, aborted(c));
      if (r == 0 && !stop)
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(peer_pfree + s * 8)
                     : "memory");
      if (stop) break;
    }
    // Epilogue: O_s = O / l, written as bf16 rows of the workspace.
    const bool done = wait_or_abort(&c->mma_done, 0, c, a.status);
    tc_fence_after();
    const int req_row = it.row0 + r;
    const bool row_ok = req_row < a.rows_per_req;
    // `done` is the same for every thread (all wait on one phase, or all see
    // the abort flag); the TMEM loads are warp-collective, the stores per row.
    if (__all_sync(0xffffffffu, done)) {
      const float inv = lfin > 0.f ? 1.f / lfin : 0.f;
      uint16_t* po = a.partial_o + ((size_t)it.slot * a.rows_per_req + (row_ok ? req_row : 0)) * kLatent;
      uint32_t v[16];
      for (int q = 0; q < 32; ++q) {
        tmem_ld16(lane_addr + 16 * q, v);
        if (row_ok) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(po + 16 * q) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(po + 16 * q + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    } else if (row_ok) {
      for (int d = 0; d < kLatent; ++d)
        a.partial_o[((size_t)it.slot * a.rows_per_req + req_row) * kLatent + d] = 0;
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const VerifyArgs a, const __grid_constant__ PoolMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Ctrl* c = reinterpret_cast<Ctrl*>(sm + BIG_END);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t role = cluster_ctarank();
  const int pair = blockIdx.x >> 1;

  Item it;
  const int row_tile = pair % a.row_tiles;
  it.slot = pair / a.row_tiles;
  const bool have = locate_split(a, it.slot, it.loc);
  it.row0 = row_tile * ROWS;
  it.k_begin = have ? it.loc.s * a.chunk_keys : 0;
  it.k_end = have ? min(it.k_begin + a.chunk_keys, it.loc.nkeys) : 0;
  it.ntiles = have ? (it.k_end - it.k_begin + TK - 1) / TK : 0;
  // Both CTAs of a cluster see the same item; an empty item skips all work
  // but still takes part in the cluster barriers.

  if (tid == 0) {
    for (int i = 0; i < QRING; ++i) { mbar_init(&c->kfull[i], 32 * kScorerProducers); mbar_init(&c->kempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->sfull[i], 1);
      mbar_init(&c->sempty[i], 4);
      mbar_init(&c->pfree[i], 2);
      mbar_init(&c->pfull[i], 1);
      mbar_init(&c->pvdone[i], 1);
    }
    for (int i = 0; i < VRING; ++i) { mbar_init(&c->vfull[i], 32 * kAccProducers); mbar_init(&c->vempty[i], 1); }
    mbar_init(&c->corr_done, 4);
    mbar_init(&c->mma_done, 1);
    c->abort = 0;
    fence_mbar_init();
  }
  if (warp == 3) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  if (role == 0 && have && tid < a.n_nodes) c->par[tid] = __ldg(a.tree_parent + (size_t)it.loc.b * a.n_nodes + tid);
  __syncthreads();
  if (role == 0 && have) {
    const int T = a.n_nodes;
    if (tid < T) c->anc[tid] = ancestor_bits_smem(c->par, tid, T, a.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (role == 0 && have && warp >= 4 && warp < 8) {
    // Q rows -> TMEM (warps 4..7, thread = query row = TMEM lane): latent as
    // packed bf16 pairs; rope -> shared memory.
    const int r = tid - 128;
    const int req_row = it.row0 + r;
    const bool ok = req_row < a.rows_per_req;
    const size_t g = (size_t)it.loc.b * a.rows_per_req + req_row;
    const uint4* ql = reinterpret_cast<const uint4*>(a.q_latent + g * a.q_lat_stride);
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)((warp - 4) * 32) << 16);
    for (int q = 0; q < 16; ++q) {  // 16 x 16 columns = 512 bf16
      uint32_t v[16];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint4 x = ok ? __ldg(ql + 4 * q + e) : make_uint4(0, 0, 0, 0);
        v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
      }
      tmem_st16(lane_addr + 16 * q, v);
    }
    tmem_st_wait();
    const uint4* qr = reinterpret_cast<const uint4*>(a.q_rope + g * a.q_rope_stride);
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
      uint4 x = ok ? __ldg(qr + c16) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sm + Q_ROPE + r * 128 + ((c16 ^ (r & 7)) << 4)) = x;
    }
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers initialised before any remote traffic

  if (have && it.ntiles > 0) {
    if (role == 0) scorer(a, maps, it, sm, c);
    else accumulator(a, maps, it, sm, c);
  }

  tc_fence_before();
  __syncthreads();
  // Tensor-core work of this CTA must be finished before TMEM is freed.
  if (warp == 3 && have && it.ntiles > 0) {
    mbar_wait(&c->mma_done, 0, kWaitNs);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote copy or arrival may target a CTA that has exited
  tc_fence_after();
  if (warp == 3) tmem_dealloc(c->tmem_base, 512);
}

}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library does not link libcuda directly).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// Pool maps over [rows, 576] bf16 with 1152-byte rows.  With an unknown pool
// size the row extent is the int32 index range (the caller vouches for the
// indices); otherwise rows past the pool read as zeros.
cudaError_t make_pool_maps(const VerifyArgs& a, PoolMaps* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t rows = a.pool_rows > 0 ? (cuuint64_t)a.pool_rows : (cuuint64_t)0x7fffffff;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  const cuuint32_t box4[2] = {64, 1}, boxt[2] = {64, 128}, es[2] = {1, 1};
  void* base = const_cast<uint16_t*>(a.kv_pool);
  if (enc(&m->row4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box4, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (enc(&m->tile, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, boxt, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace

namespace {
// The kernel needs more than the default 48 KB of dynamic shared memory;
// the attribute is set once per device.
cudaError_t ensure_smem_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_partial_tc(const VerifyArgs& a, cudaStream_t stream) {
  PoolMaps maps;
  cudaError_t e = make_pool_maps(a, &maps);
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr();
  if (e != cudaSuccess) return e;
  dim3 grid(2 * a.row_tiles * a.total_splits);
  partial_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

// How many 2-CTA clusters of this kernel the current device runs at
// once.  Clusters are placed within one GPC, so this can be below SMs / 2.
cudaError_t cluster_capacity_tc(int* clusters) {
  cudaError_t e = ensure_smem_attr();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(2 * 64);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  return cudaOccupancyMaxActiveClusters(clusters, (void*)partial_tc_kernel, &cfg);
}

}  // namespace ddtree
