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
// memory; S tiles (128 rows x 128 keys, fp32) double-buffered in TMEM; two
// softmax warpgroups (one query row per thread, 64 keys each) mask tree keys
// against the ancestor bits, agree on a lazily rescaled running max and write
// P (bf16, K-major, 128-byte swizzle) plus per-row rescale factors, shipped
// to the same-row-tile accumulator by a bulk shared-memory copy.
// Accumulator CTA: O (128 x 512 fp32) in all 512 TMEM columns; its epilogue
// warps rescale O rows when the running max moved (rare) and finally write
// O_s = O / l; the scorer writes lse_s.
//
// Gathers ("Chunk 66.1": 128-bit KV loads): the work item's indices pass
// through a shared-memory ring filled ahead by a loader warp.  Load/store-
// unit warps copy the scattered 1152-byte rows as 64-column chunks with
// 16-byte cp.async (measured faster per SM than TMA gather4 for these rows);
// a tile whose 128 indices form one contiguous run comes by 2-D TMA tile
// loads instead.  TMA loads complete on the stream's own barriers (one warp
// issues; a lane of a load/store-unit warp waits for each unit's bytes and
// counts the stream in), so every load a CTA issued is known to have landed
// before it exits, also after an expired wait.  No warp runs two spinning
// roles: a lane suspended in a barrier wait holds back every other lane of
// its warp.  The scorer's key ring holds seven units of three chunks (2.3
// tiles), enough to keep the next tile's rows in flight while a tile is
// multiplied.  The follower CTA of each pair forwards "my unit is complete"
// to the leader, whose MMA threads (one per S buffer) issue each unit's MMAs
// as soon as the unit is complete in both CTAs.
//
// Merge ("Chunk 66.0": partial + reduce): with a one-wave plan the launch is
// cooperative and the kernel merges its own splits.  Each CTA counts 2 at a
// grid barrier (release reductions) as soon as its own writes are done (an
// accumulator's two epilogue store threads once their TMA stores complete;
// every other CTA before the cluster teardown), and polls the count.  Then
// each CTA merges two rows of a request from TMA tile loads of all their
// splits.  A request with a single split needs no merge: its work item writes
// the final rows itself and the merge skips it.
//
// Every mbarrier wait is bounded; on expiry the kernel sets
// DDTREE_ST_TIMEOUT, stops issuing work, waits (bounded) for its own
// tensor-core work and frees its TMEM.
#include <cuda.h>
#include <string.h>

#include "combine.cuh"
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
// Scorer ring: units of three chunks of its 64 keys (tile t = units 3t ..
// 3t+2; chunk c of a unit at c x 8 KB), seven unit slots.  Accumulator ring:
// whole tiles of its 4 value chunks of all 128 keys (chunk q = columns
// 64 (2q+p) .. at q x 16 KB), two slots.
constexpr int QUNIT = 3 * SCHUNK;        // 24 KB
constexpr int QSLOTS = 7;
constexpr int VSLOT = 4 * VCHUNK;        // 64 KB
constexpr int VSLOTS = 2;
constexpr int kMaxSlots = QSLOTS;
constexpr int PTILE = 32768;             // bf16 P tile: 2 swizzle atoms of 128 rows x 128 B
constexpr int META = 1552;               // alpha[128], l0[128], l1[128], flag words[4]
constexpr int PCOPY = PTILE + META;      // bytes shipped per tile (multiple of 16)
constexpr int PBUF = 34816;              // P buffer stride (1024-aligned)
constexpr int NIDX = 8;                  // index ring: tiles of indices held ahead
constexpr int kThreads = 512;            // 16 warps
// Producer warps on the load/store unit (cp.async): the gather rate of an SM
// grows with the warps issuing (about 18 / 33 / 47 GB/s per SM with 4 / 8 / 16
// warps in a probe), so every warp a role can spare gathers.
constexpr int kScLsuWarps = 4;           // scorer CTAs
constexpr int kAccLsuWarps = 8;          // accumulator CTAs
__host__ __device__ constexpr int lsu_warps(uint32_t rank) { return rank < 2 ? kScLsuWarps : kAccLsuWarps; }
constexpr int kLoaderWarp = 15;
constexpr float kLazyRescale = 8.0f;     // rescale only when the max grows by > 2^8 (log2 units)
// Tensor-core work must be complete before TMEM is freed: this wait keeps a
// fixed bound whatever the caller's limit.
constexpr uint64_t kDrainNs = 2000000000ull;
constexpr uint16_t kScorerPair = 0x3, kAccPair = 0xC;

// Shared-memory map (offsets from a 1024-aligned base).
constexpr int Q_ROPE = 0;                               // scorer: 16 KB
constexpr int Q_RING = Q_ROPE + VCHUNK;                 // scorer: 7 x 24 KB
constexpr int Q_STAGE = Q_RING + QSLOTS * QUNIT;        // scorer: P staging
constexpr int Q_END = Q_STAGE + PBUF;
// Q latent (128 rows x 512 bf16, eight 64-column 128-byte-swizzled boxes)
// lands by TMA in ring slots 3.. and most of the P staging buffer, before
// any of them is used (the first tile's three units need only slots 0..2);
// the softmax warps move it into TMEM.
constexpr int kQStageSlot = 3;
constexpr int Q_LAT_STAGE = Q_RING + kQStageSlot * QUNIT;
constexpr int Q_LAT_BYTES = ROWS * kLatent * 2;
constexpr int Q_ROPE_BYTES = ROWS * kRope * 2;
static_assert(Q_LAT_STAGE + Q_LAT_BYTES <= Q_END, "Q latent staging fits the unused ring");
static_assert(Q_LAT_STAGE % 1024 == 0, "128-byte swizzle wants 1024-byte aligned boxes");
constexpr int V_PBUF = 0;                               // accumulator: 2 x PBUF
constexpr int V_RING = V_PBUF + 2 * PBUF;               // accumulator: 2 x 64 KB
constexpr int V_END = V_RING + VSLOTS * VSLOT;
static_assert(VSLOTS * VSLOT >= 8 * ROWS * 128, "the epilogue's eight 16 KB boxes fit the value ring");
constexpr int IDX_RING = (Q_END > V_END ? Q_END : V_END);  // both: NIDX x 128 int32
constexpr int BIG_END = IDX_RING + NIDX * TK * 4;


struct __align__(8) Ctrl {
  // Ring slot barriers (per unit slot): full = this CTA's chunks of the unit
  // landed (every load/store-unit lane + the TMA stream), peer = (leader)
  // the follower's slot is full, empty = the pair's MMAs consumed the slot
  // (commit multicast to both CTAs of the pair); tma = the TMA stream's
  // loads of the unit landed.
  uint64_t full[kMaxSlots], peer[kMaxSlots], empty[kMaxSlots], tma[kMaxSlots];
  // scorer
  uint64_t sfull[2], sempty[2], pfree[2];
  // accumulator
  uint64_t pfull[2], pvdone[2], corr_done[2];
  // both
  uint64_t ifull[NIDX], iempty[NIDX];  // index ring
  int32_t ifirst[NIDX];    // first index of each ring tile
  int32_t icontig[NIDX];   // the tile's 128 indices form one run
  uint64_t mma_done;
  uint64_t q_ready;   // scorer: Q latent in TMEM and Q rope in shared memory
  uint64_t qload;     // scorer: the TMA loads of Q (latent staging + rope) landed
  uint64_t mload;     // fused merge: a unit's partials landed
  uint64_t wait_ns;        // bound of the waits (the caller's, default 2 s)
  uint32_t tmem_base;
  uint32_t abort;
  alignas(16) float xmax[2][128];  // scorer: per-row maxima / sums exchanged between the softmax halves
  uint32_t merge_zero;     // fused merge: the partials cannot be trusted (a wait timed out)
  uint32_t grid_arrived;   // fused merge: grid-barrier arrivals already made by the epilogue
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
// Bounded wait on a barrier phase; on expiry mark the CTA aborted.  False
// when aborted.  CTA-scope acquire also for the barriers that other CTAs of
// the cluster arrive on: what they announce is tensor-core, bulk-copy or
// cp.async work whose completion the barrier itself tracks (or a forward of
// such a completion), not generic stores of the remote thread; a
// cluster-scope acquire measured slower on these per-unit waits.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctrl* c, uint32_t* status) {
  if (aborted(c)) return false;
  if (mbar_wait(bar, parity, c->wait_ns)) return true;
  set_abort(c, status);
  return false;
}
// Arrive on a barrier in another CTA of the cluster.  Relaxed: a pure
// signal.  Every use orders what it must by other means (the data it
// announces was itself completed through an mbarrier, or is a register value
// already consumed).  Under a load of in-flight copies a cluster-scope
// release here cost up to ~1.5 us per arrive.
__device__ __forceinline__ void signal_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
// Arrive with cluster-scope release: the arriving thread's earlier shared-
// memory reads must be complete before the remote side reuses the memory.
__device__ __forceinline__ void release_remote(uint32_t remote_bar) {
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
// tensor cycles per SM, so the issue path must stay short.
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
  bool direct;   // the request's only split, merged in this launch: final rows, no partials
};

struct PoolMaps {
  CUtensorMap half;   // 64 columns x 64 rows box: a scorer's half of a contiguous tile
  CUtensorMap tile;   // 64 columns x 128 rows box: an accumulator chunk of a contiguous tile
  CUtensorMap po;     // partial O [splits][rows_per_req][512] bf16, 64 columns x 128 rows box
  CUtensorMap ql;     // Q latent [B*T*H rows][512] bf16, 64 columns x 128 rows box
  CUtensorMap qr;     // Q rope [B*T*H rows][64] bf16, 64 columns x 128 rows box
  CUtensorMap pm;     // partial O again, unswizzled box of 256 columns x 2 rows x merge_depth splits
  CUtensorMap fo;     // out as [batch][rows_per_req][512]: single-split requests' final rows
};

// The start-of-kernel cluster barrier is split: every thread arrives once its
// CTA's barriers and TMEM are set up, and a thread waits for the other CTAs
// only before its first remote action (an arrive on, a copy to, or an MMA
// reading another CTA).  Producers that touch only their own CTA start at
// once.  Every thread waits exactly once (the kernel waits for those that did
// not) before the closing cluster barrier.
__device__ __forceinline__ void join_cluster(bool& joined) {
  if (!joined) {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
    joined = true;
  }
}

// ------------------------------------------------------------ index ring
__device__ __forceinline__ int* ring_tile(uint8_t* sm, int t) {
  return reinterpret_cast<int*>(sm + IDX_RING) + (t % NIDX) * TK;
}

// Loader warp: tile j's 128 indices (invalid ones -> -1, flagged) into ring
// slot j % NIDX, with the tile's first index and whether it is one run.  The
// loads of kIdxBatch tiles go out together, each at an address clamped into
// the work item's keys (the keys past its end are masked when stored): a load
// under a condition feeding a select would wait for each in turn.  The first
// batch is issued while the CTA is still being set up.  One tile per batch
// measured fastest (batches of 1 / 2 / 4 / 8 tiles: 48.0–49.9 / 49.9 / 50.2 /
// 54.0 us on the 65k workload, 23.3 / 23.3 / 25.5 / 29.5 us on a 4k prefix):
// the loader runs ahead through the ring anyway, and a smaller batch reaches
// the first tile's indices sooner.  (An L2 prefetch of the rows from this
// warp measured slower: the prefetch instructions held the loader back.)
constexpr int kIdxBatch = 1;
__device__ __forceinline__ void index_batch_load(const VerifyArgs& a, const Item& it, int j0, int lane,
                                                 int (&v)[kIdxBatch][4]) {
#pragma unroll
  for (int jj = 0; jj < kIdxBatch; ++jj) {
    const int k0 = it.k_begin + (j0 + jj) * TK + 4 * lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[jj][e] = __ldg(a.kv_indices + it.loc.idx_base + min(k0 + e, it.k_end - 1));
  }
}
__device__ void index_loader(const VerifyArgs& a, const Item& it, uint8_t* sm, Ctrl* c,
                             const int (&first_batch)[kIdxBatch][4]) {
  constexpr int kBatch = kIdxBatch;
  const int lane = threadIdx.x & 31;
  for (int j0 = 0; j0 < it.ntiles; j0 += kBatch) {
    int v[kBatch][4];
    if (j0 == 0) {
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) v[jj][e] = first_batch[jj][e];
    } else {
      index_batch_load(a, it, j0, lane, v);
    }
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      const int j = j0 + jj, slot = j % NIDX;
      if (j >= it.ntiles) break;
      if (j >= NIDX && !wait_bar(&c->iempty[slot], ((j / NIDX) - 1) & 1, c, a.status)) return;
      const int k0 = it.k_begin + j * TK + 4 * lane;
      int* w = v[jj];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (k0 + e >= it.k_end) {
          w[e] = -1;  // past the work item's keys (the load was clamped)
        } else if (w[e] < 0 || (a.pool_rows > 0 && w[e] >= a.pool_rows)) {
          atomicOr(a.status, DDTREE_ST_BAD_INDEX);
          w[e] = -1;
        }
      }
      int* dst = ring_tile(sm, j);
      *reinterpret_cast<int4*>(dst + 4 * lane) = make_int4(w[0], w[1], w[2], w[3]);
      const int first = __shfl_sync(0xffffffffu, w[0], 0);
      const bool run = w[0] >= 0 && w[0] == first + 4 * lane && w[1] == w[0] + 1 && w[2] == w[0] + 2 &&
                       w[3] == w[0] + 3;
      const bool contig = __all_sync(0xffffffffu, run);
      if (lane == 0) {
        c->ifirst[slot] = first;
        c->icontig[slot] = contig ? 1 : 0;
      }
      __syncwarp();
      mbar_arrive(&c->ifull[slot]);  // 32 arrivals: every lane's stores are released
    }
  }
}

// Waits until ring tile t is loaded (every lane acquires it).
__device__ __forceinline__ bool wait_ring(const VerifyArgs& a, Ctrl* c, int t) {
  return wait_bar(&c->ifull[t % NIDX], (t / NIDX) & 1, c, a.status);
}
__device__ __forceinline__ void release_ring(Ctrl* c, int t, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&c->iempty[t % NIDX]);
}

// cp.async of the 64-column chunks c0 + k * cstep (k < NC; chunk k lands at
// dst + k * dst_step) of the key rows ids[j] (chunk rows row0 + 4 j + lane/8,
// j < N; row r at + 128 r, 128-byte swizzled); a missing key (-1) writes
// zeros.  Row by row: each row's pieces go out back to back, so the requests
// for one row's bytes reach memory together (measured 4 % faster on the 65k
// workload and 11 % on the mixed batch than chunk by chunk).
template <int N, int NC>
__device__ __forceinline__ void lsu_rows(const uint16_t* pool, uint8_t* dst, uint32_t dst_step, int c0, int cstep,
                                         int row0, const int (&ids)[N], int lane) {
  const int piece = lane & 7;
  const uint32_t base = smem_u32(dst);
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int row = row0 + 4 * j + (lane >> 3);
    const int id = ids[j];
    const uint16_t* src = pool + (size_t)(id < 0 ? 0 : id) * kRow + c0 * 64 + piece * 8;
#pragma unroll
    for (int k = 0; k < NC; ++k)
      cp_async16_zfill(base + k * dst_step + row * 128 + ((piece ^ (row & 7)) << 4), src + k * cstep * 64,
                       id < 0 ? 0u : 16u);
  }
}
// One 2-D TMA tile (a contiguous run of rows) of one 64-column chunk.
__device__ __forceinline__ void tma_run(const CUtensorMap* map, uint8_t* dst, int col_chunk, int first_row,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(col_chunk * 64), "r"(first_row), "r"(smem_u32(bar))
      : "memory");
}

// The TMA stream of a CTA: 2-D tile loads of the units of contiguous tiles,
// over a ring of `nslots` unit slots, `upt` units per tile.  One thread
// issues: it starts each such unit's loads once the slot is free,
// `issue(n, t, u, slot, bar)` arming the slot's barrier `bar` with the bytes.
// Lane 0 of load/store-unit warp 0 counts the stream in on the slot's full
// barrier: at once for a scattered unit (no TMA bytes), once the bytes landed
// for a contiguous one.  Both sides track the phase parity of each slot's
// TMA barrier from the same per-tile flags.  A non-null `gate` is waited for
// (phase 0) before unit kQStageSlot is loaded.  Only the last load started on a slot
// can still be in flight (an earlier one was consumed before its slot was
// reused), so before it leaves the issuer waits (fixed bound) for those.
template <typename Issue>
__device__ __forceinline__ void tma_issuer(const VerifyArgs& a, const Item& it, Ctrl* c, int upt, int nslots,
                                           uint64_t* gate, Issue&& issue) {
  uint32_t par = 0, armed = 0;  // per slot: parity of the next TMA phase; a load was started
  const int nunits = it.ntiles * upt;
  for (int n = 0; n < nunits; ++n) {
    const int t = n / upt, u = n - t * upt, slot = n % nslots;
    if (u == 0 && !wait_ring(a, c, t)) break;
    bool free = true;
    if (c->icontig[t % NIDX] != 0) {
      free = (n != kQStageSlot || gate == nullptr || wait_bar(gate, 0, c, a.status)) &&
             wait_bar(&c->empty[slot], ((n / nslots) & 1) ^ 1, c, a.status);
      if (free) {
        issue(n, t, u, slot, &c->tma[slot]);
        par ^= 1u << slot;
        armed |= 1u << slot;
      }
    }
    if (!free || u == upt - 1) mbar_arrive(&c->iempty[t % NIDX]);
    if (!free) break;
  }
  for (int slot = 0; slot < nslots; ++slot)
    if ((armed >> slot) & 1u) mbar_wait(&c->tma[slot], ((par >> slot) & 1u) ^ 1u, kDrainNs);
}
// Lane 0 of load/store-unit warp 0: count the TMA stream in on unit slot
// `slot` (see tma_issuer); `tpar` is this side's copy of the parities.
__device__ __forceinline__ bool tma_count_in(const VerifyArgs& a, Ctrl* c, bool contig, int slot, uint32_t& tpar) {
  if (contig) {
    if (!wait_bar(&c->tma[slot], (tpar >> slot) & 1u, c, a.status)) return false;
    tpar ^= 1u << slot;
  }
  mbar_arrive(&c->full[slot]);
  return true;
}

// ------------------------------------------------------------------ scorer
__device__ void scorer(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c,
                       uint32_t rank, bool& joined, const int (&first_idx)[kIdxBatch][4]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;  // [0,256): Q latent; [256,384), [384,512): S
  const bool leader = (rank & 1) == 0;
  const int half = rank & 1;           // which 64 keys of each tile this CTA gathers

  // Producer warps: load/store unit {0, 2, 3, 12}; TMA issuer 13
  // (contiguous runs).  MMA issuers (leader): 1 (even tiles), 14 (odd).
  const int lsu = warp == 0 ? 0 : warp == 2 ? 1 : warp == 3 ? 2 : warp == 12 ? 3 : -1;
  if (warp == kLoaderWarp) {
    index_loader(a, it, sm, c, first_idx);
  } else if (lsu >= 0) {
    constexpr int G = 16 / kScLsuWarps;  // groups of four keys per warp (of the half's 16)
    uint32_t tpar = 0;                 // (warp 0) TMA phase parities, see tma_issuer
    for (int t = 0; t < it.ntiles; ++t) {
      if (!wait_ring(a, c, t)) break;
      const int* keys = ring_tile(sm, t) + HALF * half;
      const bool contig = c->icontig[t % NIDX] != 0;
      int ids[G];
#pragma unroll
      for (int j = 0; j < G; ++j) ids[j] = keys[4 * (G * lsu + j) + (lane >> 3)];
      release_ring(c, t, lane);
      bool ok = true;
      for (int u = 0; u < 3 && ok; ++u) {
        const int n = 3 * t + u, slot = n % QSLOTS;
        // Slots kQStageSlot.. hold the Q latent staging until the softmax
        // warps moved it into TMEM (q_ready).
        if (lane == 0)
          ok = (n != kQStageSlot || wait_bar(&c->q_ready, 0, c, a.status)) &&
               wait_bar(&c->empty[slot], ((n / QSLOTS) & 1) ^ 1, c, a.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* unit = sm + Q_RING + slot * QUNIT;
        if (!contig) {  // a contiguous tile comes by TMA
          lsu_rows<G, 3>(a.kv_pool, unit, SCHUNK, 3 * u, 1, 4 * G * lsu, ids, lane);
        }
        cp_async_mbar_arrive(&c->full[slot]);
        if (lsu == 0) {
          if (lane == 0) ok = tma_count_in(a, c, contig, slot, tpar);
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 13 && lane == 0) {
    tma_issuer(a, it, c, 3, QSLOTS, &c->q_ready, [&](int n, int t, int u, int slot, uint64_t* bar) {
      (void)n;
      uint8_t* unit = sm + Q_RING + slot * QUNIT;
      const bool load = c->icontig[t % NIDX] != 0;
      mbar_arrive_expect_tx(bar, load ? QUNIT : 0);
      if (load)
        for (int cc = 0; cc < 3; ++cc)
          tma_run(&maps.half, unit + cc * SCHUNK, 3 * u + cc, c->ifirst[t % NIDX] + HALF * half, bar);
    });
  } else if (leader && (warp == 1 || warp == 14) && lane == 0) {
    // ---- MMA issuers for the pair, one per S buffer: warp 1 takes the even
    // tiles, warp 14 the odd ones, so one issuer's waits for its next tile
    // overlap the other's MMAs.  A tile goes out unit by unit as its units land.
    {
      constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, false);
      const uint64_t rope_desc = desc_sw128(smem_u32(sm + Q_ROPE), 16, 1024);
      const int s = warp == 1 ? 0 : 1;
      join_cluster(joined);
      bool ok = wait_bar(&c->q_ready, 0, c, a.status);
      tc_fence_after();
      for (int t = s; t < it.ntiles && ok; t += 2) {
        const uint32_t sbuf = tmem + 256 + 128 * s;
        ok = wait_bar(&c->sempty[s], ((t >> 1) & 1) ^ 1, c, a.status);
        // Each unit's MMAs go out as soon as it landed in both CTAs, so the
        // tile's first units free their ring slots while its last one is
        // still in flight (the ring's bytes in flight set the gather rate).
#pragma unroll
        for (int u = 0; u < 3 && ok; ++u) {
          const int n = 3 * t + u, slot = n % QSLOTS;
          const uint32_t ph = (n / QSLOTS) & 1;
          ok = wait_bar(&c->full[slot], ph, c, a.status) && wait_bar(&c->peer[slot], ph, c, a.status);
          if (!ok) break;
          fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
          const uint8_t* unit = sm + Q_RING + slot * QUNIT;
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {  // chunk ch = 3u + cc: K steps 4ch .. 4ch+3 of the 36
            const int ch = 3 * u + cc;
            const uint64_t kdesc = desc_sw128(smem_u32(unit + cc * SCHUNK), 16, 1024);
            if (ch < 8) mma2_ts_x4(sbuf, tmem + ch * 32, kdesc, idesc, ch > 0);  // latent: Q from TMEM
            else mma2_ss_x4<2, 2>(sbuf, rope_desc, kdesc, idesc, 1);            // rope: Q from shared memory
          }
          commit2(&c->empty[slot], kScorerPair);
        }
        if (!ok) break;
        commit2(&c->sfull[s], kScorerPair);
      }
      commit2(&c->mma_done, kScorerPair);
    }
  } else if (!leader && warp == 1 && lane == 0) {
    {
      // ---- follower: forward "my unit n is full" to the leader
      const uint32_t lead_peer = map_cluster(smem_u32(&c->peer[0]), rank - 1);
      join_cluster(joined);
      // The leader's MMAs read this CTA's Q too: it must be in place before
      // the first forward.
      if (!wait_bar(&c->q_ready, 0, c, a.status)) return;
      for (int n = 0; n < 3 * it.ntiles; ++n) {
        const int slot = n % QSLOTS;
        if (!wait_bar(&c->full[slot], (n / QSLOTS) & 1, c, a.status)) return;
        fence_async_smem();
        signal_remote(lead_peer + slot * 8);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ---- softmax: two warpgroups; thread = (query row r, key half hw)
    const int hw = warp >= 8 ? 1 : 0;
    const int w = warp & 3;
    const int r = 32 * w + lane;
    const int req_row = it.row0 + r;
    const bool row_ok = req_row < a.rows_per_req;
    const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
    {
      // Parents of the request's nodes, for the ancestor bits below.
      const int T = a.n_nodes;
      const bool owns_node = hw == 0 && r < T;
      const int par_r = owns_node ? __ldg(a.tree_parent + (size_t)it.loc.b * T + r) : 0;
      // Q latent of row r, this half's 256 values: the TMA staging (eight
      // 128-byte-swizzled 64-column boxes) -> TMEM lane r.  Q rope came by
      // TMA straight into its place.
      if (wait_bar(&c->qload, 0, c, a.status)) {
        const uint8_t* row = sm + Q_LAT_STAGE + r * 128;
#pragma unroll 1
        for (int b4 = 0; b4 < 4; ++b4) {
          const uint8_t* box = row + (4 * hw + b4) * (ROWS * 128);
          uint32_t v[2][16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // 16-byte piece j: latent columns 8j .. 8j+7 of the box
            const uint4 x = *reinterpret_cast<const uint4*>(box + ((j ^ (r & 7)) << 4));
            uint32_t* d = &v[j >> 2][4 * (j & 3)];
            d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
          }
          tmem_st16(lane_addr + 128 * hw + 32 * b4, v[0]);
          tmem_st16(lane_addr + 128 * hw + 32 * b4 + 16, v[1]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->q_ready);  // also: the staging is free for keys
      if (owns_node) c->par[r] = par_r;
      named_bar(1, 256);
      if (owns_node) c->anc[r] = ancestor_bits_smem(c->par, r, T, a.status);
      named_bar(1, 256);
    }
    join_cluster(joined);  // remote from here on: sempty arrives, P copies
    const uint64_t anc = row_ok ? c->anc[req_row / a.n_heads] : 0ull;
    const float scale2 = a.sm_scale * 1.4426950408889634f;  // scores in log2 units
    float m_ref = -INFINITY, l = 0.f;
    const uint32_t acc_rank = rank + 2;
    const uint32_t peer_pbuf = map_cluster(smem_u32(sm + V_PBUF), acc_rank);
    const uint32_t peer_pfull = map_cluster(smem_u32(&c->pfull[0]), acc_rank);
    const uint32_t lead_sempty = map_cluster(smem_u32(&c->sempty[0]), rank & ~1u);
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      const int k0 = it.k_begin + t * TK + 64 * hw;  // first key of this half
      // Valid-key bits of this half (lane j: keys j and 32 + j).
      uint32_t km[2] = {0u, 0u};
      if (wait_ring(a, c, t)) {
        const int* keys = ring_tile(sm, t) + 64 * hw;
#pragma unroll
        for (int q = 0; q < 2; ++q) km[q] = __ballot_sync(0xffffffffu, keys[32 * q + lane] >= 0);
        release_ring(c, t, lane);
      }
      wait_bar(&c->sfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      tc_fence_after();
      uint32_t xr[2][32];  // raw fp32 scores of this row, this half's 64 keys
#pragma unroll
      for (int q = 0; q < 2; ++q) tmem_ld32(lane_addr + 256 + 128 * s + 64 * hw + 32 * q, xr[q]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) signal_remote(lead_sempty + s * 8);  // S buffer s read (leader counts 16 warps)
      uint32_t mw[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
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
      if ((mw[0] & mw[1]) == 0xffffffffu) {  // all visible: no selects
#pragma unroll
        for (int k = 0; k < 64; ++k) mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(xr[k >> 5][k & 31]));
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float v = ((mw[k >> 5] >> (k & 31)) & 1u) ? __uint_as_float(xr[k >> 5][k & 31]) : -INFINITY;
          xr[k >> 5][k & 31] = __float_as_uint(v);
          mx[k & 3] = fmaxf(mx[k & 3], v);
        }
      }
      const float mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale2;
      c->xmax[hw][r] = mh;
      // The staging buffer is free once the previous tile's copy has read it.
      if (r == 0 && hw == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      named_bar(1, 256);
      const float mt = fmaxf(mh, c->xmax[hw ^ 1][r]);
      float alpha = 1.f;
      if (mt > m_ref + kLazyRescale) {  // also true on the first finite max
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
        m_ref = mt;
      }
      const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
      uint8_t* stg = sm + Q_STAGE;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {  // 16-byte chunk cc = keys 8cc .. 8cc+7 of this half
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
        *reinterpret_cast<uint4*>(stg + hw * VCHUNK + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      const float sum = (row_ok ? 1.f : 0.f) * ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      l = l * alpha + sum;
      float* meta = reinterpret_cast<float*>(stg + PTILE);
      meta[128 * (1 + hw) + r] = l;
      if (hw == 0) {
        meta[r] = alpha;
        const uint32_t flag = __ballot_sync(0xffffffffu, t > 0 && alpha != 1.f);
        if (lane == 0) reinterpret_cast<uint32_t*>(meta + 384)[w] = flag;
      }
      fence_async_smem();
      named_bar(1, 256);
      if (r == 0 && hw == 0 && !aborted(c)) {
        // The accumulator's P buffer s is free once it finished tile t-2.
        if (wait_bar(&c->pfree[s], ((t >> 1) & 1) ^ 1, c, a.status)) {
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
              "cp.async.bulk.commit_group;" ::"r"(peer_pbuf + s * PBUF),
              "r"(smem_u32(stg)), "r"(PCOPY), "r"(peer_pfull + s * 8)
              : "memory");
        }
      }
      if (named_bar_or(1, 256, aborted(c))) break;
    }
    if (hw == 1) c->xmax[1][r] = l;
    named_bar(1, 256);
    if (hw == 0 && row_ok) {
      const float lt = l + c->xmax[1][r];
      const float lse = (lt > 0.f) ? (m_ref + log2f(lt)) * 0.6931471805599453f : -INFINITY;
      if (it.direct) a.lse[(size_t)it.loc.b * a.rows_per_req + req_row] = lse;
      else a.partial_lse[(size_t)it.slot * a.rows_per_req + req_row] = lse;
    }
    if (r == 0 && hw == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

// ------------------------------------------------------------ accumulator
// Accumulator epilogue: O_s = O / l as bf16 rows of the workspace, by eight
// warps -- 4..7 (after the tile loop) write columns 0..255, 12..15 columns
// 256..511 (a warp reaches the TMEM lanes of its index mod 4).  Each
// 64-column slice goes TMEM -> registers -> its own 128-byte-swizzled 16 KB
// box in the value ring (idle once the last PV completed) -> one TMA store,
// which writes whole rows' slices coalesced and clips the rows past the
// request.
__device__ void acc_epilogue(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int w = warp & 3, r = 32 * w + lane, hc = warp >= 12 ? 1 : 0;
  const uint32_t lane_addr = c->tmem_base + ((uint32_t)(w * 32) << 16);
  named_bar(3, 256);  // warps 12..15 wait here until warps 4..7 finished the tile loop
  const bool done = wait_bar(&c->mma_done, 0, c, a.status);
  const bool all_done = !named_bar_or(3, 256, !done);
  tc_fence_after();
  if (all_done) {
    const float l = c->xmax[0][r];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    constexpr int kBox = ROWS * 128;  // 16 KB
    const bool store = w == 0 && lane == 0 && it.row0 < a.rows_per_req;
#pragma unroll 1
    for (int q = 4 * hc; q < 4 * hc + 4; ++q) {
      uint8_t* box = sm + V_RING + q * kBox;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(lane_addr + 64 * q + 32 * h, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 16-byte piece 4h + j: columns 8 (4h + j) ..
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[8 * j + 2 * e]) * inv,
                                                      __uint_as_float(v[8 * j + 2 * e + 1]) * inv);
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(box + r * 128 + (((4 * h + j) ^ (r & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      // Each box goes out as soon as its 128 threads wrote it.
      fence_async_smem();
      named_bar(4 + hc, 128);
      if (store) {
        asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                     ::"l"(it.direct ? &maps.fo : &maps.po), "r"(64 * q), "r"(it.row0),
                       "r"(it.direct ? it.loc.b : it.slot), "r"(smem_u32(box))
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    if (w == 0 && lane == 0) {
      if (store) {
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        // The stores are read by other CTAs in the fused merge.
        asm volatile("fence.proxy.async;" ::: "memory");
      }
      // This half of the CTA's partial rows is in global memory: it counts
      // itself in at the merge's grid barrier now (release), instead of after
      // the CTA's teardown.  Both halves always do, so the CTA owes none later.
      if (a.fused) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.grid_done) : "memory");
      if (hc == 0) c->grid_arrived = 2;
    }
  } else if (hc == 0 && it.row0 + r < a.rows_per_req) {
    uint16_t* dst = it.direct ? a.out + ((size_t)it.loc.b * a.rows_per_req + it.row0 + r) * kLatent
                              : a.partial_o + ((size_t)it.slot * a.rows_per_req + it.row0 + r) * kLatent;
    for (int d = 0; d < kLatent; ++d) dst[d] = 0;
  }
}

// Whether the P tile in buffer s asks for a rescale of O before its PV: the
// softmax sets a flag word per warp when the running max of a row moved.
__device__ __forceinline__ bool rescaled(const uint8_t* sm, int s) {
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(sm + V_PBUF + s * PBUF + PTILE + 384 * 4);
  return (flags[0] | flags[1] | flags[2] | flags[3]) != 0u;
}

__device__ void accumulator(const VerifyArgs& a, const PoolMaps& maps, const Item& it, uint8_t* sm, Ctrl* c,
                            uint32_t rank, bool& joined, const int (&first_idx)[kIdxBatch][4]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c->tmem_base;  // O: cols [0,512)
  const bool leader = (rank & 1) == 0;
  const int par = rank & 1;            // value chunks 2q + par of every tile
  const uint32_t scorer_rank = rank - 2;
  // Producer warps: load/store unit {0, 2, 3, 8, 9, 12, 13, 14} (12..14 then
  // join the epilogue); TMA issuer 10 (contiguous runs).  MMA issuers
  // (leader): 1 (O columns 0..255), 11 (256..511).
  const int lsu = warp == 0 ? 0 : warp == 2 ? 1 : warp == 3 ? 2 : warp == 8 ? 3 : warp == 9 ? 4
                : (warp >= 12 && warp <= 14) ? warp - 7 : -1;

  if (warp == kLoaderWarp) {
    index_loader(a, it, sm, c, first_idx);
  } else if (lsu >= 0) {
    constexpr int G = 32 / kAccLsuWarps;  // groups of four keys per warp (of the tile's 32)
    uint32_t tpar = 0;                 // (warp 0) TMA phase parities, see tma_issuer
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      if (!wait_ring(a, c, t)) break;
      const int* keys = ring_tile(sm, t);
      const bool contig = c->icontig[t % NIDX] != 0;
      int ids[G];
#pragma unroll
      for (int j = 0; j < G; ++j) ids[j] = keys[4 * (G * lsu + j) + (lane >> 3)];
      release_ring(c, t, lane);
      bool ok = true;
      if (lane == 0) ok = wait_bar(&c->empty[s], ((t >> 1) & 1) ^ 1, c, a.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* slot = sm + V_RING + s * VSLOT;
      if (!contig) {
        lsu_rows<G, 4>(a.kv_pool, slot, VCHUNK, par, 2, 4 * G * lsu, ids, lane);
      }
      cp_async_mbar_arrive(&c->full[s]);
      if (lsu == 0) {
        if (lane == 0) ok = tma_count_in(a, c, contig, s, tpar);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 10 && lane == 0) {
    tma_issuer(a, it, c, 1, VSLOTS, nullptr, [&](int n, int t, int u, int slot, uint64_t* bar) {
      (void)n;
      (void)u;
      uint8_t* dst = sm + V_RING + slot * VSLOT;
      const bool load = c->icontig[t % NIDX] != 0;
      mbar_arrive_expect_tx(bar, load ? VSLOT : 0);
      if (load)
        for (int q = 0; q < 4; ++q) tma_run(&maps.tile, dst + q * VCHUNK, 2 * q + par, c->ifirst[t % NIDX], bar);
    });
  } else if (leader && (warp == 1 || warp == 11) && lane == 0) {
    // ---- MMA issuers for the pair: O[rows, 128q .. 128q+127] += P V, warp 1
    // for q = 0, 1 and warp 11 for q = 2, 3 (disjoint accumulator columns,
    // so their MMAs need no order between them); each counts in on every
    // tile's empty / pvdone barrier.
    {
      constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, true);  // A = P K-major, B = V MN-major
      const int q0 = warp == 1 ? 0 : 2;
      join_cluster(joined);
      for (int t = 0; t < it.ntiles; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        // P and V of both CTAs in place (the follower's forward also covers
        // its own rescale); this CTA's O rescaled first when the running max
        // of any of its rows moved (flags in the P metadata).
        if (!wait_bar(&c->pfull[s], ph, c, a.status) || !wait_bar(&c->full[s], ph, c, a.status) ||
            !wait_bar(&c->peer[s], ph, c, a.status) ||
            (rescaled(sm, s) && !wait_bar(&c->corr_done[s], ph, c, a.status)))
          break;
        fence_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
        tc_fence_after();
        const uint64_t pdesc = desc_sw128(smem_u32(sm + V_PBUF + s * PBUF), 16, 1024);
        const uint8_t* slot = sm + V_RING + s * VSLOT;
#pragma unroll
        for (int q = q0; q < q0 + 2; ++q) {
          const uint64_t vdesc = desc_sw128(smem_u32(slot + q * VCHUNK), VCHUNK, 1024);
          // K steps 0..3 read P atom 0 (keys 0..63), 4..7 atom 1; V advances
          // 16 keys (2 KB) per step.
          mma2_ss_x4<2, 128>(tmem + 128 * q, pdesc, vdesc, idesc, t > 0 ? 1u : 0u);
          mma2_ss_x4<2, 128>(tmem + 128 * q, pdesc + (VCHUNK >> 4), vdesc + 512, idesc, 1u);
        }
        commit2(&c->empty[s], kAccPair);
        commit2(&c->pvdone[s], kAccPair);
        commit2(&c->pfree[s], kScorerPair);  // both scorers may refill P buffer s
      }
      commit2(&c->mma_done, kAccPair);
    }
  } else if (!leader && warp == 1 && lane == 0) {
    {
      // ---- follower: forward "my P tile and my value slot of tile t are
      // both full" to the leader, as one arrive
      const uint32_t lead_peer = map_cluster(smem_u32(&c->peer[0]), rank - 1);
      join_cluster(joined);
      for (int t = 0; t < it.ntiles; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!wait_bar(&c->pfull[s], ph, c, a.status) || !wait_bar(&c->full[s], ph, c, a.status) ||
            (rescaled(sm, s) && !wait_bar(&c->corr_done[s], ph, c, a.status)))
          return;
        fence_async_smem();
        signal_remote(lead_peer + s * 8);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---- correction (then half of the epilogue): thread = row r (TMEM lane r)
    const int r = tid - 128;
    const int w = warp - 4;
    const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
    const uint32_t sc_pfree = map_cluster(smem_u32(&c->pfree[0]), scorer_rank);
    join_cluster(joined);
    // P buffers 0 and 1 expect their first copies (later phases are armed
    // below, once the previous phase was seen complete).
    if (r == 0)
      for (int s = 0; s < 2 && s < it.ntiles; ++s) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
    float lfin = 0.f;
    for (int t = 0; t < it.ntiles; ++t) {
      const int s = t & 1;
      wait_bar(&c->pfull[s], (t >> 1) & 1, c, a.status);  // on expiry: continue, stop below
      const uint8_t* pb = sm + V_PBUF + s * PBUF;
      const float* meta = reinterpret_cast<const float*>(pb + PTILE);
      const uint32_t* flags = reinterpret_cast<const uint32_t*>(meta + 384);
      lfin = meta[128 + r] + meta[256 + r];
      if (flags[0] | flags[1] | flags[2] | flags[3]) {
        const float alpha = meta[r];
        // O must hold PV of tiles < t before it is rescaled.
        wait_bar(&c->pvdone[(t - 1) & 1], ((t - 1) >> 1) & 1, c, a.status);
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
      // Every tile: this CTA's O is ready for PV(t) (waited for only when
      // the flags asked for a rescale).
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->corr_done[s]);
      // P buffer s: its metadata has been read (the scorer's third release,
      // after the two MMA issuers' commits), and its next phase may be armed.
      const bool stop = named_bar_or(2, 128, aborted(c));
      if (r == 0 && !stop) {
        if (t + 2 < it.ntiles) mbar_arrive_expect_tx(&c->pfull[s], PCOPY);
        release_remote(sc_pfree + s * 8);
      }
      if (stop) break;
    }
    c->xmax[0][r] = lfin;  // the row's final l, for the epilogue (published by its barrier)
  }
  if ((warp >= 4 && warp < 8) || warp >= 12) acc_epilogue(a, maps, it, sm, c);
}

// ------------------------------------------------------------ fused merge
// The split merge by tile loads (after the grid barrier): a unit is two rows
// of one request; one thread loads all of the request's split partials for
// them (two boxes of 256 columns x 2 rows x merge_depth splits, 2 KB per
// split) into shared memory, two warps turn the rows' split LSEs into
// weights, and every thread merges two columns of one row:
//     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
// `zero` writes zero rows and -inf LSEs (untrusted partials).
__device__ __forceinline__ int tile_merge_units(const VerifyArgs& a) { return a.batch * ((a.rows_per_req + 1) >> 1); }
// The split range of tile-merge unit u (two rows of request u / pairs).
__device__ __forceinline__ void tile_merge_slots(const VerifyArgs& a, int u, int& first, int& count) {
  const int b = u / ((a.rows_per_req + 1) >> 1);
  combine_slots(a, b * a.rows_per_req * kCombineUnitsPerRow, threadIdx.x & 31, first, count);
}
// (first, count): the slots of this CTA's first unit, looked up in advance.
__device__ void tile_merge(const VerifyArgs& a, const PoolMaps& maps, uint8_t* sm, Ctrl* c, bool zero, int first,
                           int count) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.merge_depth;
  const int pairs = (a.rows_per_req + 1) >> 1;
  const int units = tile_merge_units(a);
  const uint32_t box_bytes = 256u * 2u * (uint32_t)D * 2u;
  float* wgt = c->xmax[0];  // [2 rows][64 splits] weights
  float* rowl = c->xmax[1]; // [2 rows]: l, then lse
  uint32_t ph = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ph ^= 1u) {
    const int b = u / pairs, r0 = 2 * (u - b * pairs);
    if (u != (int)blockIdx.x) tile_merge_slots(a, u, first, count);
    // A request's only split wrote its final rows itself (unless a wait
    // expired: then every row is zeroed here).
    if (count == 1 && !zero) {
      ph ^= 1u;  // no load this unit: undo the loop's phase step
      continue;
    }
    count = zero ? 0 : min(count, D);
    if (tid == 0 && count > 0) {
      // The partials were written by other CTAs' TMA stores, seen through
      // the grid barrier (generic proxy); these loads are async proxy.
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(&c->mload, 2 * box_bytes);
      for (int h = 0; h < 2; ++h)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
            ::"r"(smem_u32(sm + h * box_bytes)), "l"(&maps.pm), "r"(256 * h), "r"(r0), "r"(first), "r"(smem_u32(&c->mload))
            : "memory");
    }
    if (warp < 2) {  // warp w: the weights of row r0 + w (lane j: splits j, j + 32)
      const int row = r0 + warp;
      const bool live = row < a.rows_per_req;
      const float* pl = a.partial_lse + (size_t)first * a.rows_per_req + (live ? row : 0);
      // Both loads issued together at clamped addresses and masked after (a
      // load under a condition feeding a select would wait for each in
      // turn); none when the request has no splits here (its first slot may
      // then lie past the partials).
      float xa = -INFINITY, xb = -INFINITY;
      if (count > 0) {
        xa = __ldcg(pl + (size_t)min(lane, count - 1) * a.rows_per_req);
        xb = __ldcg(pl + (size_t)min(lane + 32, count - 1) * a.rows_per_req);
      }
      const float la = (live && lane < count) ? xa : -INFINITY;
      const float lb = (live && lane + 32 < count) ? xb : -INFINITY;
      float m = fmaxf(la, lb);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float wa = la == -INFINITY ? 0.f : __expf(la - m);
      const float wb = lb == -INFINITY ? 0.f : __expf(lb - m);
      float l = wa + wb;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      wgt[64 * warp + lane] = wa * inv;
      wgt[64 * warp + lane + 32] = wb * inv;
      if (lane == 0) rowl[warp] = l > 0.f ? m + logf(l) : -INFINITY;
    }
    __syncthreads();
    bool ok = true;
    if (count > 0) ok = mbar_wait(&c->mload, ph, a.wait_ns);
    if (!ok && tid == 0) atomicOr(a.status, DDTREE_ST_TIMEOUT);
    // thread: row r0 + (tid >> 8), columns 2 (tid & 255) .. + 1
    const int rr = tid >> 8, col = 2 * (tid & 255);
    const int row = r0 + rr;
    if (row < a.rows_per_req) {
      const int h = col >> 8;
      const uint8_t* src = sm + h * box_bytes + rr * 512 + (col & 255) * 2;
      // Four splits per step into two sums of each column (the loads of a
      // step are independent; the chains are half as long).
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      if (ok) {
        const float* wr = wgt + 64 * rr;
        int s = 0;
#pragma unroll 1
        for (; s + 4 <= count; s += 4) {
          const float4 w = *reinterpret_cast<const float4*>(wr + s);  // one load for four weights
          uint32_t x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = *reinterpret_cast<const uint32_t*>(src + (size_t)(s + e) * 1024);
          acc0 = fmaf(w.x, bf16_lo(x[0]), acc0);
          acc1 = fmaf(w.x, bf16_hi(x[0]), acc1);
          acc2 = fmaf(w.y, bf16_lo(x[1]), acc2);
          acc3 = fmaf(w.y, bf16_hi(x[1]), acc3);
          acc0 = fmaf(w.z, bf16_lo(x[2]), acc0);
          acc1 = fmaf(w.z, bf16_hi(x[2]), acc1);
          acc2 = fmaf(w.w, bf16_lo(x[3]), acc2);
          acc3 = fmaf(w.w, bf16_hi(x[3]), acc3);
        }
        for (; s < count; ++s) {
          const uint32_t x = *reinterpret_cast<const uint32_t*>(src + (size_t)s * 1024);
          acc0 = fmaf(wr[s], bf16_lo(x), acc0);
          acc1 = fmaf(wr[s], bf16_hi(x), acc1);
        }
      }
      acc0 += acc2;
      acc1 += acc3;
      const size_t g = (size_t)b * a.rows_per_req + row;
      *reinterpret_cast<__nv_bfloat162*>(a.out + g * kLatent + col) = __floats2bfloat162_rn(acc0, acc1);
      if ((tid & 255) == 0) a.lse[g] = ok ? rowl[rr] : -INFINITY;
    }
    __syncthreads();  // the boxes and weights are reused by the next unit
    if (count == 0) ph ^= 1u;  // no load this unit: the barrier did not move
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
  // A request with one split needs no merge: with the merge in this launch,
  // its work item writes the final O and LSE rows itself.
  it.direct = have && a.fused && it.loc.ns == 1;
  // All four CTAs see the same key range; an empty item skips all work but
  // still takes part in the cluster barriers and the pair's TMEM allocation.

  const bool work = have && it.ntiles > 0;
  // The loader warp's first index loads, in flight during the set-up below.
  int first_idx[kIdxBatch][4];
  if (warp == kLoaderWarp && work) index_batch_load(a, it, 0, tid & 31, first_idx);
  if (tid == 0) {
    for (int i = 0; i < kMaxSlots; ++i) {
      mbar_init(&c->full[i], 32 * lsu_warps(rank) + 1);  // every load/store-unit lane, the TMA stream
      mbar_init(&c->peer[i], 1);
      mbar_init(&c->empty[i], rank < 2 ? 1 : 2);  // accumulator: both MMA issuers commit
      mbar_init(&c->tma[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->sfull[i], 1);
      mbar_init(&c->sempty[i], 16);
      mbar_init(&c->pfree[i], 3);  // two PV commits + the metadata release
      mbar_init(&c->pfull[i], 1);
      mbar_init(&c->pvdone[i], 2);
      mbar_init(&c->corr_done[i], 4);
    }
    // Index ring: the loader's 32 lanes fill a slot; it is released by every
    // producer warp, and in the scorers also by the eight softmax warps.
    for (int i = 0; i < NIDX; ++i) {
      mbar_init(&c->ifull[i], 32);
      mbar_init(&c->iempty[i], lsu_warps(rank) + 1 + (rank < 2 ? 8 : 0));
    }
    mbar_init(&c->mma_done, 2);  // two MMA issuers per pair
    mbar_init(&c->q_ready, 8);
    mbar_init(&c->qload, 1);
    mbar_init(&c->mload, 1);
    c->abort = 0;
    c->grid_arrived = 0;
    c->wait_ns = a.wait_ns;
    fence_mbar_init();
    if (rank < 2 && work) {
      // The scorer's Q first: latent into the staging, rope into place.
      const int g0 = it.loc.b * a.rows_per_req + it.row0;
      mbar_arrive_expect_tx(&c->qload, Q_LAT_BYTES + Q_ROPE_BYTES);
      for (int b = 0; b < kLatent / 64; ++b) tma_run(&maps.ql, sm + Q_LAT_STAGE + b * (ROWS * 128), b, g0, &c->qload);
      tma_run(&maps.qr, sm + Q_ROPE, 0, g0, &c->qload);
    }
  }
  if (warp == 3) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&c->tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // This CTA's barriers and TMEM are ready for the others; each thread waits
  // for theirs before its first remote action (join_cluster).  Relaxed: the
  // barrier initialisation was published by its own fence, and nothing else
  // written so far is read by another CTA.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  bool joined = false;
  if (work) {
    if (rank < 2) scorer(a, maps, it, sm, c, rank, joined, first_idx);
    else accumulator(a, maps, it, sm, c, rank, joined, first_idx);
  }
  join_cluster(joined);
  // The Q loads have landed before the CTA leaves (also after an expired wait).
  if (tid == 0 && rank < 2 && work) mbar_wait(&c->qload, 0, kDrainNs);

  tc_fence_before();
  __syncthreads();
  if (a.fused && tid == 0) {
    // Fused merge: every CTA counts 2 at the grid barrier.  An accumulator's
    // epilogue did so as soon as its partial rows were stored; the rest
    // count here, as soon as the CTA's own writes (LSEs, zero rows) are done,
    // without waiting for the rest of the cluster.  Release: those writes,
    // ordered before this thread by the barrier above, are visible to
    // whoever sees the count.
    const uint32_t late = 2u - c->grid_arrived;
    if (late) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.grid_done), "r"(late) : "memory");
  }
  // Tensor-core work writing this CTA's TMEM must be finished before it is freed.
  if (warp == 3 && work) mbar_wait_cluster(&c->mma_done, 0, kDrainNs);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote copy or arrival may target a CTA that has exited
  tc_fence_after();
  if (warp == 3)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(c->tmem_base), "r"(512) : "memory");

  if (a.fused) {
    // Merge the splits in this launch: every CTA of the grid is resident at
    // once (cooperative launch), so each, having counted itself in above,
    // waits, bounded, for all others; then each CTA merges two rows at a
    // time from one tile load of all their splits (the plan fuses only when
    // a request's splits fit it).  A timed-out wait anywhere writes zeros.
    // The split range of the CTA's first unit, looked up while the grid finishes.
    int first = 0, count = 0;
    if ((int)blockIdx.x < tile_merge_units(a)) tile_merge_slots(a, blockIdx.x, first, count);
    if (tid == 0) {
      uint64_t deadline = 0;
      bool ok = true;
      for (uint32_t spin = 1;; ++spin) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.grid_done) : "memory");
        if (v >= 2u * gridDim.x) break;
        if (spin == 4u) {
          deadline = global_timer_ns() + a.wait_ns;
        } else if (spin > 4u && (spin & 7u) == 0u && global_timer_ns() > deadline) {
          ok = false;
          break;
        }
      }
      if (!ok) atomicOr(a.status, DDTREE_ST_TIMEOUT);
      uint32_t st;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(st) : "l"(a.status) : "memory");
      c->merge_zero = (!ok || (st & DDTREE_ST_TIMEOUT)) ? 1u : 0u;
    }
    __syncthreads();
    tile_merge(a, maps, sm, c, c->merge_zero != 0, first, count);
  }
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
// half).  Rows past the pool read as zeros; with
// an unknown pool size the row extent is the int32 index range (the caller
// vouches for the indices).
cudaError_t make_pool_maps(const VerifyArgs& a, PoolMaps* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t rows = a.pool_rows > 0 ? (cuuint64_t)a.pool_rows : (cuuint64_t)0x7fffffff;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  const cuuint32_t box_half[2] = {64, (cuuint32_t)HALF}, box_tile[2] = {64, (cuuint32_t)TK};
  const cuuint32_t es[2] = {1, 1};
  void* base = const_cast<uint16_t*>(a.kv_pool);
  const cuuint32_t* boxes[2] = {box_half, box_tile};
  CUtensorMap* maps[2] = {&m->half, &m->tile};
  for (int i = 0; i < 2; ++i)
    if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, boxes[i], es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  // Partial O: [total_splits][rows_per_req][512] bf16; rows past the request
  // fall outside dimension 1, so a store of a partial row tile is clipped.
  const cuuint64_t odims[3] = {(cuuint64_t)kLatent, (cuuint64_t)a.rows_per_req, (cuuint64_t)a.total_splits};
  const cuuint64_t ostrides[2] = {(cuuint64_t)kLatent * 2, (cuuint64_t)a.rows_per_req * kLatent * 2};
  const cuuint32_t obox[3] = {64, (cuuint32_t)ROWS, 1}, oes[3] = {1, 1, 1};
  if (enc(&m->po, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.partial_o, odims, ostrides, obox, oes,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // The fused merge's view of the partials: two rows x 256 columns of up to
  // merge_depth consecutive splits per box (splits past the last read zeros).
  if (a.merge_depth > 0) {
    const cuuint32_t mbox[3] = {256, 2, (cuuint32_t)a.merge_depth};
    if (enc(&m->pm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.partial_o, odims, ostrides, mbox, oes,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Final output as [batch][rows_per_req][512] bf16, for single-split
  // requests that write their rows directly (rows past a request clipped).
  if (a.fused) {
    const cuuint64_t fdims[3] = {(cuuint64_t)kLatent, (cuuint64_t)a.rows_per_req, (cuuint64_t)a.batch};
    if (enc(&m->fo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.out, fdims, ostrides, obox, oes,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Queries: rows (t, h) of all requests, request-major; rows past the last
  // one read as zeros.  The row strides are multiples of 8 elements and the
  // bases 16-byte aligned (checked when the call is validated).
  const cuuint64_t qrows = (cuuint64_t)a.batch * (cuuint64_t)a.rows_per_req;
  const cuuint64_t qldims[2] = {(cuuint64_t)kLatent, qrows}, qlstr[1] = {(cuuint64_t)a.q_lat_stride * 2};
  const cuuint64_t qrdims[2] = {(cuuint64_t)kRope, qrows}, qrstr[1] = {(cuuint64_t)a.q_rope_stride * 2};
  const cuuint32_t qbox[2] = {64, (cuuint32_t)ROWS};
  if (enc(&m->ql, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.q_latent), qldims, qlstr, qbox,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&m->qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.q_rope), qrdims, qrstr, qbox,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
  if (!a.fused) {
    partial_tc2_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, maps);
    return cudaGetLastError();
  }
  // The fused merge waits on every CTA of the grid: a cooperative launch
  // guarantees they are all resident (or fails to launch).
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, partial_tc2_kernel, a, maps);
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

