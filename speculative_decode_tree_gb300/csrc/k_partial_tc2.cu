// Split-KV partial stage on tcgen05 tensor cores, CTA-pair (cta_group::2) form.
//
// One work item = two 128-row tiles of one request (rows 256*p .. 256*p+255)
// x one chunk of the request's key sequence ("Chunk 66.0": KV-split flash
// decode, partial + reduce; the split count is the plan's, "Chunk 66.1"),
// run by a cluster of four CTAs:
//
//   rank 0, 1  scorer pair      (row tile 2p, 2p+1)   S = Q K^T, softmax -> P
//   rank 2, 3  accumulator pair (row tile 2p, 2p+1)   O += P V
//
// The pairs issue M = 256 MMAs with cta_group::2: the even rank of each pair
// issues them for both, each CTA holds the A operand and the D accumulator of
// its own 128 rows, and the B operand is split between the two CTAs' shared
// memory.  So each key tile is gathered ONCE per pair: scorer CTA c loads
// keys 64c .. 64c+63 of every 128-key tile (all 576 columns), accumulator CTA
// 2+c loads value chunks 2q+c (64 of the 512 columns) of all 128 keys.
//
// Scorer CTA: Q latent (128 x 512 bf16) in TMEM (A operand), Q rope in shared
// memory; S tiles (128 rows x 128 keys, fp32) double-buffered in TMEM; four
// softmax warps (one query row per thread) mask tree keys against the
// ancestor bits, keep a lazily rescaled running max and write P (bf16,
// K-major, 128-byte swizzle) plus per-row rescale factors, shipped to the
// same-row-tile accumulator by a bulk shared-memory copy across the cluster.
// Accumulator CTA: O (128 x 512 fp32) in all 512 TMEM columns; its epilogue
// warps rescale O rows when the running max moved (rare) and finally write
// O_s = O / l; the scorer writes lse_s.
//
// Gathers: 16-byte cp.async of the scattered 1152-byte rows through the
// page_size=1 index table ("Chunk 66.1": 128-bit KV loads) into 128-byte
// swizzled chunks; a tile whose 128 indices form one contiguous run uses 2-D
// TMA tile loads instead.  The follower CTA of each pair forwards "my half
// landed" to the leader, whose MMA thread waits for both halves.
//
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

constexpr int TK = 128;                  // keys per tile
constexpr int ROWS = 128;                // query rows per CTA
constexpr int HALF = 64;                 // keys per scorer CTA per tile
constexpr int SCHUNK = HALF * 128;       // scorer chunk: 64 keys x 64 columns (8 KB)
constexpr int VCHUNK = TK * 128;         // accumulator chunk: 128 keys x 64 columns (16 KB)
// The key rings are rings of units of several chunks with one mbarrier per
// unit: a producer warp signals a unit with one cp.async-tracked arrive, which
// keeps more bytes in flight per arrive than a barrier per chunk.
constexpr int QU = 3;                    // scorer chunks per unit (24 KB)
constexpr int QUNITS = 7;                // scorer unit slots (2.3 tiles)
constexpr int QUNIT_BYTES = QU * SCHUNK;
constexpr int VU = 2;                    // accumulator chunks per unit (32 KB)
constexpr int VUNITS = 4;                // accumulator unit slots (2 tiles)
constexpr int VUNIT_BYTES = VU * VCHUNK;
constexpr int PTILE = 32768;             // bf16 P tile: 2 swizzle atoms of 128 rows x 128 B
constexpr int META = 1040;               // alpha[128], lfin[128], flag words[4]
constexpr int PCOPY = PTILE + META;      // bytes shipped per tile (multiple of 16)
constexpr int PBUF = 34816;              // P buffer stride (1024-aligned)
constexpr int kThreads = 384;            // 12 warps
constexpr int kScorerProducers = 7;      // warps 0, 2, 3, 8..11
constexpr int kAccProducers = 6;         // warps 0, 3, 8..11
constexpr int kScorerLsuChunks = 6;      // scorer chunks 0..5 by cp.async, 6..8 by TMA gather4
constexpr int kAccLsuChunks = 3;         // accumulator chunks q = 0..2 by cp.async, q = 3 by TMA gather4
constexpr float kLazyRescale = 8.0f;     // rescale only when the max grows by > 2^8 (log2 units)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint16_t kScorerPair = 0x3, kAccPair = 0xC;

// Shared-memory map (offsets from a 1024-aligned base).
constexpr int Q_ROPE = 0;                          // scorer: 16 KB
constexpr int Q_RING = Q_ROPE + VCHUNK;            // scorer: 7 x 24 KB
constexpr int Q_STAGE = Q_RING + QUNITS * QUNIT_BYTES;  // scorer: P staging
constexpr int Q_END = Q_STAGE + PBUF;
constexpr int V_PBUF = 0;                          // accumulator: 2 x PBUF
constexpr int V_RING = V_PBUF + 2 * PBUF;          // accumulator: 8 x 16 KB
constexpr int V_END = V_RING + VUNITS * VUNIT_BYTES;
constexpr int BIG_END = (Q_END > V_END ? Q_END : V_END);

struct __align__(8) Ctrl {
  // scorer
  uint64_t kfull[QUNITS], kpeer[QUNITS], kempty[QUNITS];
  uint64_t sfull[2], sempty[2], pfree[2];
  // accumulator
  uint64_t vfull[VUNITS], vpeer[VUNITS], vempty[VUNITS];
  uint64_t pfull[2], ppeer[2], pvdone[2], corr_done[2];
  // both
  uint64_t mma_done;
  uint64_t q_ready;   // scorer: Q latent in TMEM and Q rope in shared memory
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t key_mask[2][4];
  uint64_t anc[64];
  int32_t par[64];   // the request's parents, staged for the ancestor walk
};

constexpr size_t kSmemBytes = 1024 + BIG_END + sizeof(Ctrl) + 64;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ bool aborted(Ctrl* c) { return *(volatile uint32_t*)&c->abort != 0; }
__device__ __forceinline__ void set_abort(Ctrl* c, uint32_t* status) {
  c->abort = 1;
  atomicOr(status, DDTREE_ST_TIMEOUT);
}
// Bounded wait with cluster-scope acquire (most barriers here are arrived on
// by another CTA: peer forwards, multicast commits, bulk-copy completions);
// on expiry mark the CTA aborted.  False when aborted.
__device__ __forceinline__ bool wait_clu(uint64_t* bar, uint32_t parity, Ctrl* c, uint32_t* status) {
  if (aborted(c)) return false;
  if (mbar_wait_cluster(bar, parity, global_timer_ns() + kWaitNs)) return true;
  set_abort(c, status);
  return false;
}
__device__ __forceinline__ void remote_arrive(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
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

// ---- cta_group::2 tensor-core instructions (issued by the pair's even CTA)
// Four K steps (K = 16 each) of one 64-column chunk per statement, the
// operand addresses stepped inside PTX.  One MMA of M = 256, N = 128 is 64
// tensor cycles per SM, so the issue path must stay short: with one statement
// and C++ descriptor arithmetic per MMA the pipe ran at about 55 % on the
// 65k-prefix workload, which this form lifts by ~6 us per call.
// A from TMEM (row r in lane r, 8 columns = 16 bf16 per K step), B by
// descriptor (K-major, 128-byte swizzle: 32 bytes per K step).
__device__ __forceinline__ void mma2_ts_x4(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc,
                                           uint32_t acc_first) {
  asm volatile(
      "{ .reg .pred p; .reg .b32 a1, a2, a3; .reg .b64 b1, b2, b3;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  add.u32 a1, %1, 8; add.u32 a2, %1, 16; add.u32 a3, %1, 24;\n"
      "  add.u64 b1, %2, 2; add.u64 b2, %2, 4; add.u64 b3, %2, 6;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], [a1], b1, %3, 1;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], [a2], b2, %3, 1;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], [a3], b3, %3, 1; }" ::"r"(d),
      "r"(a0), "l"(b0), "r"(idesc), "r"(acc_first)
      : "memory");
}
// A and B both by descriptor; the descriptors advance by ASTEP / BSTEP
// (16-byte units) per K step.
template <int ASTEP, int BSTEP>
__device__ __forceinline__ void mma2_ss_x4(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc,
                                           uint32_t acc_first) {
  asm volatile(
      "{ .reg .pred p; .reg .b64 a1, a2, a3, b1, b2, b3;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  add.u64 a1, %1, %5; add.u64 a2, %1, %6; add.u64 a3, %1, %7;\n"
      "  add.u64 b1, %2, %8; add.u64 b2, %2, %9; add.u64 b3, %2, %10;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, 1;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], a2, b2, %3, 1;\n"
      "  tcgen05.mma.cta_group::2.kind::f16 [%0], a3, b3, %3, 1; }" ::"r"(d),
      "l"(a0), "l"(b0), "r"(idesc), "r"(acc_first), "n"(ASTEP), "n"(2 * ASTEP), "n"(3 * ASTEP), "n"(BSTEP),
      "n"(2 * BSTEP), "n"(3 * BSTEP)
      : "memory");
}
// Arrive once on `bar` (same offset) in every CTA of `mask` when all MMAs
// issued so far by this thread have completed.
__device__ __forceinline__ void commit2(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

struct Item {
  SplitLoc loc;
  int row0;      // first query row of this CTA's tile within the request
  int k_begin;   // first key of the chunk
  int k_end;     // one past the last key
  int ntiles;
  int slot;      // split slot in the workspace
};

struct PoolMaps {
  CUtensorMap half;   // 64 columns x 64 rows box: a scorer's half of a contiguous tile
  CUtensorMap tile;   // 64 columns x 128 rows box: an accumulator chunk of a contiguous tile
  CUtensorMap po;     // partial O [splits][rows_per_req][512] fp32, 32 columns x 128 rows box
  CUtensorMap row;    // 64 columns x 1 row box: four scattered rows per gather4 load
};

// One tile's 128 indices: lane l holds keys 4l .. 4l+3 (-1 past the chunk or
// outside the pool); the raw loads are issued a tile early.
struct RawIdx {
  int v[4];
};
struct TileIdx {
  int4 k4;
  int first;
  bool contiguous;
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

// Index of key (4 g + lane/8) of the groups this producer lane copies: a
// contiguous block of groups g = first .. first+n-1 (of ngroups, split as
// evenly as the np producer warps allow), taken from the lane that holds them
// (tile key 4 (g0 + g) + lane/8, g0 = first group of this CTA's keys).
struct MyKeys {
  int id[6];
  int n;
  int first;
};
__device__ __forceinline__ MyKeys my_keys(const TileIdx& ti, int lane, int rank, int np, int g0, int ngroups) {
  MyKeys mk;
  const int per = ngroups / np, extra = ngroups % np;
  mk.first = rank * per + min(rank, extra);
  mk.n = per + (rank < extra ? 1 : 0);
  const int sel = lane >> 3;
#pragma unroll
  for (int j = 0; j < 6; ++j) {
    const int g = mk.first + j;
    const int src = (g0 + g) & 31;
    const int x = __shfl_sync(0xffffffffu, ti.k4.x, src);
    const int y = __shfl_sync(0xffffffffu, ti.k4.y, src);
    const int z = __shfl_sync(0xffffffffu, ti.k4.z, src);
    const int w = __shfl_sync(0xffffffffu, ti.k4.w, src);
    mk.id[j] = sel == 0 ? x : sel == 1 ? y : sel == 2 ? z : w;
  }
  return mk;
}

// Fills one 64-column chunk (columns 64*col_chunk ..) of `nkeys` key rows
// (tile keys key0 .. key0+nkeys-1) into `dst` (row k at dst + 128 k,
// 128-byte swizzled).  TMA bytes are expected on `bar`; the caller arrives
// on it once per lane after the last chunk of a unit.  Scattered rows come
// by 16-byte cp.async (load/store unit) or, when `g4` is set, by TMA gather4
// loads of four rows each: the TMA engine is a second path into shared
// memory, so giving it some of the chunks raises a CTA's gather rate.
__device__ __forceinline__ void fill_chunk(const PoolMaps& maps, const uint16_t* pool, uint8_t* dst, int col_chunk,
                                           int key0, int nkeys, const TileIdx& ti, const MyKeys& mk, int rank,
                                           int lane, uint64_t* bar, bool g4) {
  if (ti.contiguous) {
    if (rank == 0 && lane == 0) {
      mbar_expect_tx(bar, nkeys * 128);
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(smem_u32(dst)), "l"(nkeys == TK ? &maps.tile : &maps.half), "r"(col_chunk * 64),
            "r"(ti.first + key0), "r"(smem_u32(bar))
          : "memory");
    }
    __syncwarp();
  } else if (g4) {
    if (lane == 0 && mk.n > 0) mbar_expect_tx(bar, mk.n * 512);
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      if (j < mk.n) {  // warp-uniform
        // Rows of group first+j are held by lanes 0, 8, 16, 24; a missing
        // key (-1) reads row 0 instead: its score is masked and its weight is 0.
        const int r0 = max(mk.id[j], 0);
        const int r1 = max(__shfl_sync(0xffffffffu, mk.id[j], 8), 0);
        const int r2 = max(__shfl_sync(0xffffffffu, mk.id[j], 16), 0);
        const int r3 = max(__shfl_sync(0xffffffffu, mk.id[j], 24), 0);
        if (lane == 0)
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst + 4 * (mk.first + j) * 128)),
              "l"(&maps.row), "r"(col_chunk * 64), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
              : "memory");
      }
    }
    __syncwarp();
  } else {
    const int piece = lane & 7;
    const uint32_t base = smem_u32(dst);
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      if (j < mk.n) {
        const int row = 4 * (mk.first + j) + (lane >> 3);  // row within this chunk
        const int id = mk.id[j];
        const uint16_t* src = pool + (size_t)(id < 0 ? 0 : id) * kRow + col_chunk * 64 + piece * 8;
        cp_async16_zfill(base + row * 128 + ((piece ^ (row & 7)) << 4), src, id < 0 ? 0u : 16u);
      }
    }
  }
}

// Pulls whole 1152-byte key rows of a tile into L2 (one bulk prefetch per
// row, from the accumulator's otherwise idle TMA unit); thread r -> key r.
// Eight tiles ahead of the accumulator (about six ahead of the scorer's
// gathers) measured best on the 65k-prefix and mixed-batch workloads: 3
// tiles ahead cost 2 us per call more, 16 (the whole chunk up front) 5 us.
constexpr int kL2Ahead = 8;
__device__ __forceinline__ void prefetch_tile_l2(const VerifyArgs& a, const Item& it, int tile, int r) {
  if (tile >= it.ntiles) return;
  const int kp = it.k_begin + tile * TK + r;
  if (kp >= it.k_end) return;
  const int id = __ldg(a.kv_indices + it.loc.idx_base + kp);
  if (id < 0 || (a.pool_rows > 0 && id >= a.pool_rows)) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.kv_pool + (size_t)id * kRow), "r"(kRow * 2)
               : "memory");
}

__device__ __forceinline__ int scorer_producer_rank(int warp) {
  if (warp == 0) return 0;
  if (warp == 2) return 1;
  if (warp == 3) return 2;
  if (warp >= 8) return warp - 5;
  return -1;
}
__device__ __forceinline__ int acc_producer_rank(int warp) {
  if (warp == 0) return 0;
  if (warp == 3) return 1;
  if (warp >= 8) return warp - 6;
  return -1;
}

// ------------------------------------------------------------------ scorer
__device__ void scorer(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c,
                       uint32_t rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;  // [0,256): Q latent; [256,384), [384,512): S
  const bool leader = (rank & 1) == 0;
  const int half = rank & 1;           // which 64 keys of each tile this CTA gathers
  const int prank = scorer_producer_rank(warp);

  if (prank >= 0) {
    // ---- producers: this CTA's 64 keys, columns 0..575, of every tile
    int n = 0;
    RawIdx raw_next = raw_tile_indices(a, it, 0, lane);
    for (int t = 0; t < it.ntiles; ++t) {
      const TileIdx ti = finish_tile_indices(a, raw_next, lane);
      if (t + 1 < it.ntiles) raw_next = raw_tile_indices(a, it, t + 1, lane);
      const MyKeys mk = my_keys(ti, lane, prank, kScorerProducers, 16 * half, 16);
      for (int u = 0; u < 9 / QU; ++u, ++n) {
        const int slot = n % QUNITS;
        bool ok = true;
        if (lane == 0) ok = wait_clu(&c->kempty[slot], ((n / QUNITS) & 1) ^ 1, c, a.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          return;
        }
#pragma unroll 1
        for (int cc = 0; cc < QU; ++cc)
          fill_chunk(maps, a.kv_pool, sm + Q_RING + slot * QUNIT_BYTES + cc * SCHUNK, QU * u + cc, HALF * half, HALF,
                     ti, mk, prank, lane, &c->kfull[slot], QU * u + cc >= kScorerLsuChunks);
        cp_async_mbar_arrive(&c->kfull[slot]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1 && lane == 0) {
    if (leader) {
      // ---- MMA issuer for the pair
      constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, false);
      const uint64_t rope_desc = desc_sw128(smem_u32(sm + Q_ROPE), 16, 1024);
      int n = 0;
      bool ok = wait_clu(&c->q_ready, 0, c, a.status);
      tc_fence_after();
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int s = t & 1;
        const uint32_t sbuf = tmem + 256 + 128 * s;
        if (!wait_clu(&c->sempty[s], ((t >> 1) & 1) ^ 1, c, a.status)) { ok = false; break; }
        tc_fence_after();
        for (int u = 0; u < 9 / QU; ++u, ++n) {
          const int slot = n % QUNITS;
          const uint32_t ph = (n / QUNITS) & 1;
          if (!wait_clu(&c->kfull[slot], ph, c, a.status) || !wait_clu(&c->kpeer[slot], ph, c, a.status)) {
            ok = false;
            break;
          }
          fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < QU; ++cc) {  // chunk ch: K steps 4ch .. 4ch+3 of the 36
            const int ch = QU * u + cc;
            const uint64_t kdesc = desc_sw128(smem_u32(sm + Q_RING + slot * QUNIT_BYTES + cc * SCHUNK), 16, 1024);
            if (ch < 8) mma2_ts_x4(sbuf, tmem + ch * 32, kdesc, idesc, ch > 0);  // latent: Q from TMEM
            else mma2_ss_x4<2, 2>(sbuf, rope_desc, kdesc, idesc, 1);            // rope: Q from shared memory
          }
          commit2(&c->kempty[slot], kScorerPair);
        }
        if (ok) commit2(&c->sfull[s], kScorerPair);
      }
      commit2(&c->mma_done, kScorerPair);
    } else {
      // ---- follower: forward "my half of unit n landed" to the leader
      const uint32_t lead_kpeer = map_cluster(smem_u32(&c->kpeer[0]), rank - 1);
      // The leader's MMAs read this CTA's Q too: it must be in place before
      // the first forward.
      if (!wait_clu(&c->q_ready, 0, c, a.status)) return;
      int n = 0;
      for (int t = 0; t < it.ntiles; ++t) {
        for (int u = 0; u < 9 / QU; ++u, ++n) {
          const int slot = n % QUNITS;
          if (!wait_clu(&c->kfull[slot], (n / QUNITS) & 1, c, a.status)) return;
          fence_async_smem();
          remote_arrive(lead_kpeer + slot * 8);
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---- softmax: thread = query row r of this CTA's tile
    const int r = tid - 128;
    const int w = warp - 4;
    const int req_row = it.row0 + r;
    const bool row_ok = req_row < a.rows_per_req;
    {
      // First, this row of Q into place while the producers already gather
      // keys: latent -> TMEM lane r as packed bf16 pairs, rope -> shared
      // memory (K-major, 128-byte swizzle).  16 loads in flight per thread.
      const size_t g = (size_t)it.loc.b * a.rows_per_req + (row_ok ? req_row : 0);
      const uint4* ql = reinterpret_cast<const uint4*>(a.q_latent + g * a.q_lat_stride);
      const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
#pragma unroll 1
      for (int b4 = 0; b4 < 4; ++b4) {
        uint4 x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = row_ok ? __ldg(ql + 16 * b4 + e) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t v[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[4 * e] = x[4 * q + e].x; v[4 * e + 1] = x[4 * q + e].y;
            v[4 * e + 2] = x[4 * q + e].z; v[4 * e + 3] = x[4 * q + e].w;
          }
          tmem_st16(lane_addr + 64 * b4 + 16 * q, v);
        }
      }
      const uint4* qr = reinterpret_cast<const uint4*>(a.q_rope + g * a.q_rope_stride);
      uint4 y[8];
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) y[c16] = row_ok ? __ldg(qr + c16) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4*>(sm + Q_ROPE + r * 128 + ((c16 ^ (r & 7)) << 4)) = y[c16];
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->q_ready);
    }
    const uint64_t anc = row_ok ? c->anc[req_row / a.n_heads] : 0ull;
    const float scale2 = a.sm_scale * 1.4426950408889634f;  // scores in log2 units
    float m_ref = -INFINITY, l = 0.f;
    const uint32_t my_lane_addr = (uint32_t)(w * 32) << 16;
    const uint32_t acc_rank = rank + 2;
    const uint32_t peer_pbuf = map_cluster(smem_u32(sm + V_PBUF), acc_rank);
    const uint32_t peer_pfull = map_cluster(smem_u32(&c->pfull[0]), acc_rank);
    const uint32_t lead_sempty = map_cluster(smem_u32(&c->sempty[0]), rank & ~1u);
    // Index of this lane's key in the next tile (warp w covers keys
    // 32w .. 32w+31), loaded one tile ahead so the load is off the loop's path.
    auto tile_has_key = [&](int tile) { return tile < it.ntiles && it.k_begin + tile * TK + 32 * w + lane < it.k_end; };
    auto tile_key_index = [&](int tile) {
      return tile_has_key(tile) ? __ldg(a.kv_indices + it.loc.idx_base + it.k_begin + tile * TK + 32 * w + lane) : -1;
    };
    int id_next = tile_key_index(0);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      const int k0 = it.k_begin + t * TK;
      {  // valid-key bits of this tile
        const int id = id_next;
        id_next = tile_key_index(t + 1);
        bool v = false;
        if (tile_has_key(t)) {
          v = id >= 0 && (a.pool_rows <= 0 || id < a.pool_rows);
          if (!v) atomicOr(a.status, DDTREE_ST_BAD_INDEX);
        }
        const uint32_t bits = __ballot_sync(0xffffffffu, v);
        if (lane == 0) c->key_mask[s][w] = bits;
      }
      wait_clu(&c->sfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      tc_fence_after();
      uint32_t xr[4][32];  // raw fp32 scores of this row, 128 keys
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tmem + my_lane_addr + 256 + 128 * s + 32 * q, xr[q]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) remote_arrive(lead_sempty + s * 8);  // S buffer s read (leader counts 8 warps)
      named_bar(1, 128);
      uint32_t km[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) km[q] = c->key_mask[s][q];
      // Visible keys of this row as 4 x 32 bits: a valid index, and for a
      // tree key (position P + j) node j must be an ancestor of the row's
      // node (or the node itself).  One select per score applies the mask.
      uint32_t mw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t bits = row_ok ? km[q] : 0u;
        const int lo = k0 + 32 * q - it.loc.P;  // tree index of key 32q (negative: prefix)
        if (lo > -32) {
          uint32_t tree;
          if (lo >= 0) tree = lo < 64 ? (uint32_t)(anc >> lo) : 0u;
          else tree = (uint32_t)(anc << (-lo)) | ((1u << (-lo)) - 1u);
          bits &= tree;
        }
        mw[q] = bits;
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        const float v = ((mw[k >> 5] >> (k & 31)) & 1u) ? __uint_as_float(xr[k >> 5][k & 31]) : -INFINITY;
        xr[k >> 5][k & 31] = __float_as_uint(v);
        mx[k & 3] = fmaxf(mx[k & 3], v);
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale2;
      float alpha = 1.f;
      if (mt > m_ref + kLazyRescale) {  // also true on the first finite max
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
        m_ref = mt;
      }
      const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // The staging buffer is free once the previous tile's copy has read it.
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
        *reinterpret_cast<uint4*>(stg + atom * VCHUNK + r * 128 + ((c16 ^ (r & 7)) << 4)) =
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
        // The accumulator's P buffer s is free once it finished tile t-2.
        if (wait_clu(&c->pfree[s], ((t >> 1) & 1) ^ 1, c, a.status)) {
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
__device__ void accumulator(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c,
                            uint32_t rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;  // O: cols [0,512)
  const bool leader = (rank & 1) == 0;
  const int par = rank & 1;            // value chunks 2q + par of every tile
  const uint32_t scorer_rank = rank - 2;
  const int prank = acc_producer_rank(warp);

  if (prank >= 0) {
    // ---- producers: value chunks 2q+par (q = 0..3), all 128 keys
    int n = 0;
    RawIdx raw_next = raw_tile_indices(a, it, 0, lane);
    for (int t = 0; t < it.ntiles; ++t) {
      const TileIdx ti = finish_tile_indices(a, raw_next, lane);
      if (t + 1 < it.ntiles) raw_next = raw_tile_indices(a, it, t + 1, lane);
      const MyKeys mk = my_keys(ti, lane, prank, kAccProducers, 0, 32);
      for (int u = 0; u < 4 / VU; ++u, ++n) {
        const int slot = n % VUNITS;
        bool ok = true;
        if (lane == 0) ok = wait_clu(&c->vempty[slot], ((n / VUNITS) & 1) ^ 1, c, a.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          return;
        }
#pragma unroll 1
        for (int cc = 0; cc < VU; ++cc)
          fill_chunk(maps, a.kv_pool, sm + V_RING + slot * VUNIT_BYTES + cc * VCHUNK, 2 * (VU * u + cc) + par, 0, TK,
                     ti, mk, prank, lane, &c->vfull[slot], VU * u + cc >= kAccLsuChunks);
        cp_async_mbar_arrive(&c->vfull[slot]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1 && lane == 0) {
    if (leader) {
      // ---- MMA issuer for the pair: O[rows, 128q .. 128q+127] += P V
      constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, true);  // A = P K-major, B = V MN-major
      int n = 0;
      bool ok = true;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!wait_clu(&c->pfull[s], ph, c, a.status) || !wait_clu(&c->ppeer[s], ph, c, a.status) ||
            !wait_clu(&c->corr_done[s], ph, c, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t pdesc = desc_sw128(smem_u32(sm + V_PBUF + s * PBUF), 16, 1024);
        for (int u = 0; u < 4 / VU; ++u, ++n) {
          const int slot = n % VUNITS;
          const uint32_t vph = (n / VUNITS) & 1;
          if (!wait_clu(&c->vfull[slot], vph, c, a.status) || !wait_clu(&c->vpeer[slot], vph, c, a.status)) {
            ok = false;
            break;
          }
          fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < VU; ++cc) {
            const int q = VU * u + cc;
            const uint64_t vdesc = desc_sw128(smem_u32(sm + V_RING + slot * VUNIT_BYTES + cc * VCHUNK), VCHUNK, 1024);
            // K steps 0..3 read P atom 0 (keys 0..63), 4..7 atom 1; V advances
            // 16 keys (2 KB) per step.
            mma2_ss_x4<2, 128>(tmem + 128 * q, pdesc, vdesc, idesc, t > 0 ? 1u : 0u);
            mma2_ss_x4<2, 128>(tmem + 128 * q, pdesc + (VCHUNK >> 4), vdesc + 512, idesc, 1u);
          }
          commit2(&c->vempty[slot], kAccPair);
        }
        if (ok) commit2(&c->pvdone[s], kAccPair);
      }
      commit2(&c->mma_done, kAccPair);
    } else {
      // ---- follower: forward "my P tile / my value chunk landed" to the leader
      const uint32_t lead_ppeer = map_cluster(smem_u32(&c->ppeer[0]), rank - 1);
      const uint32_t lead_vpeer = map_cluster(smem_u32(&c->vpeer[0]), rank - 1);
      int n = 0;
      for (int t = 0; t < it.ntiles; ++t) {
        const int s = t & 1;
        if (!wait_clu(&c->pfull[s], (t >> 1) & 1, c, a.status)) return;
        remote_arrive(lead_ppeer + s * 8);
        for (int u = 0; u < 4 / VU; ++u, ++n) {
          const int slot = n % VUNITS;
          if (!wait_clu(&c->vfull[slot], (n / VUNITS) & 1, c, a.status)) return;
          fence_async_smem();
          remote_arrive(lead_vpeer + slot * 8);
        }
      }
    }
  } else if (warp == 2 && lane == 0) {
    // ---- relay: PV of tile t finished -> re-arm P buffer s, release it to the scorer
    const uint32_t sc_pfree = map_cluster(smem_u32(&c->pfree[0]), scorer_rank);
    for (int s = 0; s < 2; ++s) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      if (!wait_clu(&c->pvdone[s], (t >> 1) & 1, c, a.status)) break;
      if (t + 2 < it.ntiles) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
      remote_arrive(sc_pfree + s * 8);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---- correction + epilogue: thread = row r (TMEM lane r)
    const int r = tid - 128;
    const int w = warp - 4;
    const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
    const uint32_t sc_pfree = map_cluster(smem_u32(&c->pfree[0]), scorer_rank);
    const uint32_t lead_corr = map_cluster(smem_u32(&c->corr_done[0]), rank & ~1u);
    float lfin = 0.f;
    for (int t = 0; t < kL2Ahead; ++t) prefetch_tile_l2(a, it, t, r);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      prefetch_tile_l2(a, it, t + kL2Ahead, r);
      wait_clu(&c->pfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      const uint8_t* pb = sm + V_PBUF + s * PBUF;
      const float* meta = reinterpret_cast<const float*>(pb + PTILE);
      const uint32_t* flags = reinterpret_cast<const uint32_t*>(meta + 256);
      lfin = meta[128 + r];
      if (flags[0] | flags[1] | flags[2] | flags[3]) {
        const float alpha = meta[r];
        // O must hold PV of tiles < t before it is rescaled.
        wait_clu(&c->pvdone[(t - 1) & 1], ((t - 1) >> 1) & 1, c, a.status);
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {  // warp-collective TMEM access
          uint32_t v[16];
#pragma unroll 1
          for (int q = 0; q < 32; ++q) {
            tmem_ld16(lane_addr + 16 * q, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(lane_addr + 16 * q, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
      }
      // Every tile: this CTA's O is ready for PV(t) (the leader counts 8 warps).
      __syncwarp();
      if (lane == 0) remote_arrive(lead_corr + s * 8);
      // Second release of P buffer s: its metadata has been read.
      const bool stop = named_bar_or(2, 128, aborted(c));
      if (r == 0 && !stop) remote_arrive(sc_pfree + s * 8);
      if (stop) break;
    }
    // Epilogue: O_s = O / l, written as fp32 rows of the workspace.  Each
    // 32-column slice of the tile goes TMEM -> registers -> a swizzled
    // shared-memory box (4 rotating 16 KB boxes in the free value ring) ->
    // one TMA store, which writes whole rows' slices coalesced and clips
    // the rows past the request.
    const bool done = wait_clu(&c->mma_done, 0, c, a.status);
    tc_fence_after();
    const int req_row = it.row0 + r;
    const bool row_ok = req_row < a.rows_per_req;
    if (__all_sync(0xffffffffu, done)) {
      const float inv = lfin > 0.f ? 1.f / lfin : 0.f;
      const bool store = it.row0 < a.rows_per_req;
      constexpr int kBox = ROWS * 128;  // 16 KB
      for (int q = 0; q < kLatent / 32; ++q) {
        uint8_t* box = sm + V_RING + (q & 3) * kBox;
        if (q >= 4) {
          // The store issued from this box four slices ago must have read it.
          if (r == 0) asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
          named_bar(2, 128);
        }
        uint32_t v[32];
        tmem_ld32(lane_addr + 32 * q, v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(box + r * 128 + ((j ^ (r & 7)) << 4)) =
              make_float4(__uint_as_float(v[4 * j]) * inv, __uint_as_float(v[4 * j + 1]) * inv,
                          __uint_as_float(v[4 * j + 2]) * inv, __uint_as_float(v[4 * j + 3]) * inv);
        fence_async_smem();
        named_bar(2, 128);
        if (r == 0 && store) {
          asm volatile(
              "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n"
              "cp.async.bulk.commit_group;" ::"l"(&maps.po), "r"(32 * q), "r"(it.row0), "r"(it.slot),
              "r"(smem_u32(box))
              : "memory");
        }
      }
      if (r == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    } else if (row_ok) {
      for (int d = 0; d < kLatent; ++d)
        a.partial_o[((size_t)it.slot * a.rows_per_req + req_row) * kLatent + d] = 0.f;
    }
  }
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc2_kernel(const VerifyArgs a, const __grid_constant__ PoolMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Ctrl* c = reinterpret_cast<Ctrl*>(sm + BIG_END);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int quad = blockIdx.x >> 2;
  const int row_pairs = (a.row_tiles + 1) >> 1;

  Item it;
  const int row_pair = quad % row_pairs;
  it.slot = quad / row_pairs;
  const bool have = locate_split(a, it.slot, it.loc);
  it.row0 = (2 * row_pair + (int)(rank & 1)) * ROWS;  // may lie past the request: all rows masked
  it.k_begin = have ? it.loc.s * a.chunk_keys : 0;
  it.k_end = have ? min(it.k_begin + a.chunk_keys, it.loc.nkeys) : 0;
  it.ntiles = have ? (it.k_end - it.k_begin + TK - 1) / TK : 0;
  // All four CTAs see the same key range; an empty item skips all work but
  // still takes part in the cluster barriers and the pair's TMEM allocation.

  if (tid == 0) {
    for (int i = 0; i < QUNITS; ++i) {
      mbar_init(&c->kfull[i], 32 * kScorerProducers);
      mbar_init(&c->kpeer[i], 1);
      mbar_init(&c->kempty[i], 1);
    }
    for (int i = 0; i < VUNITS; ++i) {
      mbar_init(&c->vfull[i], 32 * kAccProducers);
      mbar_init(&c->vpeer[i], 1);
      mbar_init(&c->vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->sfull[i], 1);
      mbar_init(&c->sempty[i], 8);
      mbar_init(&c->pfree[i], 2);
      mbar_init(&c->pfull[i], 1);
      mbar_init(&c->ppeer[i], 1);
      mbar_init(&c->pvdone[i], 1);
      mbar_init(&c->corr_done[i], 8);
    }
    mbar_init(&c->mma_done, 1);
    mbar_init(&c->q_ready, 4);
    c->abort = 0;
    fence_mbar_init();
  }
  if (warp == 3) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&c->tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (rank < 2 && have && tid < a.n_nodes) c->par[tid] = __ldg(a.tree_parent + (size_t)it.loc.b * a.n_nodes + tid);
  __syncthreads();
  if (rank < 2 && have) {
    const int T = a.n_nodes;
    if (tid < T) c->anc[tid] = ancestor_bits_smem(c->par, tid, T, a.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  cluster_sync();  // all four CTAs' barriers and TMEM ready before any remote traffic

  if (have && it.ntiles > 0) {
    if (rank < 2) scorer(a, maps, it, sm, c, rank);
    else accumulator(a, maps, it, sm, c, rank);
  }

  tc_fence_before();
  __syncthreads();
  // Tensor-core work writing this CTA's TMEM must be finished before it is freed.
  if (warp == 3 && have && it.ntiles > 0) mbar_wait_cluster(&c->mma_done, 0, global_timer_ns() + kWaitNs);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote copy or arrival may target a CTA that has exited
  tc_fence_after();
  if (warp == 3)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(c->tmem_base), "r"(512) : "memory");
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// Pool maps over [rows, 576] bf16 with 1152-byte rows, 128-byte swizzle:
// `tile` has a 128-row box (a whole tile), `half` a 64-row box (one scorer
// half).  Rows past the pool read as zeros; with an unknown pool size the
// row extent is the int32 index range (the caller vouches for the indices).
cudaError_t make_pool_maps(const VerifyArgs& a, PoolMaps* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t rows = a.pool_rows > 0 ? (cuuint64_t)a.pool_rows : (cuuint64_t)0x7fffffff;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  const cuuint32_t box_half[2] = {64, (cuuint32_t)HALF}, box_tile[2] = {64, (cuuint32_t)TK}, es[2] = {1, 1};
  void* base = const_cast<uint16_t*>(a.kv_pool);
  if (enc(&m->half, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box_half, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (enc(&m->tile, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box_tile, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const cuuint32_t box_row[2] = {64, 1};
  if (enc(&m->row, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box_row, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // Partial O: [total_splits][rows_per_req][512] fp32; rows past the request
  // fall outside dimension 1, so a store of a partial row tile is clipped.
  const cuuint64_t odims[3] = {(cuuint64_t)kLatent, (cuuint64_t)a.rows_per_req, (cuuint64_t)a.total_splits};
  const cuuint64_t ostrides[2] = {(cuuint64_t)kLatent * 4, (cuuint64_t)a.rows_per_req * kLatent * 4};
  const cuuint32_t obox[3] = {32, (cuuint32_t)ROWS, 1}, oes[3] = {1, 1, 1};
  if (enc(&m->po, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.partial_o, odims, ostrides, obox, oes,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
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
    e = cudaFuncSetAttribute(partial_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_partial_tc2(const VerifyArgs& a, cudaStream_t stream) {
  PoolMaps maps;
  cudaError_t e = make_pool_maps(a, &maps);
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr();
  if (e != cudaSuccess) return e;
  const int row_pairs = (a.row_tiles + 1) / 2;
  dim3 grid(4 * row_pairs * a.total_splits);
  partial_tc2_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

// How many 4-CTA clusters of this kernel the current device runs at
// once.  Clusters are placed within one GPC, so this can be below SMs / 4.
cudaError_t cluster_capacity_tc2(int* clusters) {
  cudaError_t e = ensure_smem_attr();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(4 * 64);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  return cudaOccupancyMaxActiveClusters(clusters, (void*)partial_tc2_kernel, &cfg);
}

}  // namespace ddtree
