/*
 * ddtree_verify.h — C ABI of the DDTree verify-attention library (sm_103a).
 *
 * The operation.  DDTree speculative decoding scores every node of a draft
 * token tree in one target-model forward ("verify").  In MLA absorbed form,
 * every (node i, head h) query row of 576 bf16 values (512 latent + 64 rope)
 * attends over
 *     K(i) = the request's P prefix tokens  u  the tree nodes on the path from
 *            i up to its root (i included),
 * where each key is one 576-wide bf16 row of a token-granular (page_size=1)
 * KV pool reached through an int32 index table, and the value is the first
 * 512 columns of that same row:
 *     s_k  = sm_scale * <q[i,h], pool[k]>,  O[i,h] = sum_k softmax(s)_k pool[k,:512],
 *     LSE[i,h] = ln sum_k exp(s_k).
 * Sources: magik.net "Chunk 66.0" (verify attention on MLA with page_size=1,
 * scattered KV at ~14 GB/s; the KV-split flash-decode "partial+reduce" kernel)
 * and "Chunk 66.1" (the capture-safe rewrite: static buffers, no host syncs,
 * copies or cudaMalloc, a fixed split count, a torch-allocated workspace;
 * NSPLIT raised 16 -> 64 for the 8-heads-per-rank regime; 128-bit KV loads).
 *
 * Conventions shared by every entry point
 *  - Pointers named q_*, kv_*, tree_parent, prefix_lens, out, lse, workspace
 *    are DEVICE pointers; *_host pointers are host pointers.
 *  - bf16 tensors are passed as raw 16-bit patterns (ddtree_bf16_t).
 *  - Ownership: the caller owns every buffer, including the workspace.  The
 *    library allocates nothing at run time and keeps no global state beyond
 *    a per-device cache of the SM count and compute capability; its device
 *    image holds one fixed scratch array (DDTREE_NOALLOC_SCRATCH_BYTES, used
 *    only by ddtree_verify_mla_noalloc) on every GPU that loads it.  All device work is
 *    enqueued on the caller's `stream`; there is no host synchronisation
 *    (except in ddtree_verify_mla_check, by design), so calls can be
 *    captured into a CUDA graph.  `out` and `lse` are fully overwritten.
 *  - Return codes: DDTREE_OK or a DDTREE_E* code.  Argument errors are found
 *    on the host before anything is enqueued.  Bad DEVICE data (an index
 *    outside the pool, a parent that is not -1 or an earlier node, lengths
 *    beyond the plan) is never dereferenced: the kernels drop the offending
 *    key or work item and OR a bit into the status word at the start of the
 *    workspace, which ddtree_verify_mla_check reads.  Kernels never trap.
 */
#ifndef DDTREE_VERIFY_H
#define DDTREE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DDTREE_API __attribute__((visibility("default")))
#else
#define DDTREE_API
#endif

typedef uint16_t ddtree_bf16_t;      /* raw bf16 bits */
struct CUstream_st;                  /* cudaStream_t == struct CUstream_st* */
struct CUevent_st;                   /* cudaEvent_t  == struct CUevent_st*  */

#define DDTREE_LATENT_DIM 512
#define DDTREE_ROPE_DIM 64
#define DDTREE_ROW_DIM 576           /* 1152 bytes per KV row */
#define DDTREE_MAX_NODES 64          /* ancestor sets are one 64-bit mask */
#define DDTREE_MAX_HEADS 128
#define DDTREE_MAX_BATCH 1024

enum ddtree_status {
  DDTREE_OK = 0,
  DDTREE_EINVAL = 1,        /* null/misaligned pointer or out-of-range size   */
  DDTREE_EWORKSPACE = 2,    /* workspace smaller than the plan needs          */
  DDTREE_EUNSUPPORTED = 3,  /* no sm_103 / sm_100 device current             */
  DDTREE_ELAUNCH = 4,       /* a kernel launch failed (cudaGetLastError)      */
  DDTREE_EDEVICE_DATA = 5,  /* ddtree_verify_mla_check: status word non-zero  */
  DDTREE_ECUDA = 6          /* another CUDA runtime error                    */
};

/* Bits of the device status word (workspace offset 0, uint32). */
#define DDTREE_ST_BAD_INDEX   0x1u   /* kv_indices entry < 0 or >= pool_rows  */
#define DDTREE_ST_BAD_PARENT  0x2u   /* parent not -1 and not an earlier node */
#define DDTREE_ST_BAD_LENGTH  0x4u   /* device lengths exceed the plan        */
#define DDTREE_ST_TIMEOUT     0x8u   /* a bounded wait in a kernel expired    */
#define DDTREE_ST_OVERLAP     0x10u  /* relocation: a destination row is busy  */
#define DDTREE_ST_BAD_MASK    0x20u  /* a custom mask that is not a tree mask  */

/* Kernel variants of the split-KV partial stage. */
#define DDTREE_KERNEL_AUTO 0
#define DDTREE_KERNEL_SIMT 1         /* CUDA-core partial kernel              */
#define DDTREE_KERNEL_TC   2         /* tcgen05 / TMEM partial kernel, CTA pair per 128-row tile */
#define DDTREE_KERNEL_TC2  3         /* tcgen05 cta_group::2 kernel, 4-CTA cluster per 256 rows  */

/*
 * Execution plan: every size the launch needs, fixed on the host so the grid
 * does not depend on device data (capture-safe, "Chunk 66.1": fixed NSPLIT).
 * Split rule ("Chunk 66.1": NSPLIT 16 -> 64 because 8 heads per rank left the
 * GPU starved): each request's key sequence (P_b prefix keys, then T tree
 * keys) is cut into chunks of `chunk_keys`; one chunk of one row tile is one
 * work item; `chunk_keys` is chosen so that work items fill the SMs.
 * Fields are outputs of ddtree_verify_mla_plan except the two q strides and
 * wait_limit_us, which the caller may set afterwards (0 = contiguous rows,
 * 0 = the default 2 s bound).
 */
typedef struct ddtree_plan {
  int32_t batch;            /* B                                              */
  int32_t n_nodes;          /* T, the same for every request (1..64)          */
  int32_t n_heads;          /* H (1..128)                                     */
  int32_t rows_per_req;     /* T*H query rows per request                     */
  int64_t pool_rows;        /* KV pool rows (index bound); <= 0: unchecked    */
  int32_t max_keys;         /* max_b (P_b + T) of the planned lengths         */
  int32_t kernel;           /* DDTREE_KERNEL_SIMT, _TC or _TC2                */
  int32_t tile_keys;        /* keys per inner tile                            */
  int32_t chunk_keys;       /* keys per split (multiple of tile_keys)         */
  int32_t total_splits;     /* sum_b ceil((P_b+T)/chunk_keys), planned        */
  int32_t row_tile;         /* query rows per work item                       */
  int32_t row_tiles;        /* ceil(rows_per_req / row_tile)                  */
  int32_t num_sms;          /* SMs the plan spreads its work items over       */
  int32_t q_latent_row_stride; /* elements between (t,h) rows; 0 -> 512       */
  int32_t q_rope_row_stride;   /* elements between (t,h) rows; 0 -> 64        */
  int64_t workspace_bytes;  /* bytes the workspace must hold                  */
  int64_t off_partial_lse;  /* byte offsets inside the workspace: fp32 LSEs   */
  int64_t off_partial_o;    /*   [splits, rows], bf16 partial O [splits, rows, 512] */
  int32_t fused_combine;    /* 1: the partial kernel merges the splits itself
                               (cluster-of-four kernel, every cluster resident
                               at once: a cooperative launch); 0: a separate
                               combine kernel follows                       */
  int32_t wait_limit_us;    /* bound of each wait inside the cluster-of-four
                               kernel, in microseconds; 0 = 2 s.  A wait that
                               expires sets DDTREE_ST_TIMEOUT and the call
                               finishes with zero outputs (caller-settable,
                               e.g. to test that path)                      */
  int32_t reserved[6];
} ddtree_plan_t;

/*
 * Make a plan for `batch` requests of `n_nodes` tree nodes and `n_heads`
 * heads with prefix lengths prefix_lens_host[0..batch) (host array).  The
 * plan is an upper bound: a later call may use shorter device lengths (e.g.
 * graph replay), never longer ones.  pool_rows bounds kv_indices (<= 0
 * disables the check).  Host-only apart from cached device queries (SM
 * count, and how many clusters of the chosen kernel are resident at once).
 * Errors: DDTREE_EINVAL (sizes out of range, null pointers),
 * DDTREE_EUNSUPPORTED (no CUDA device to size for).
 */
DDTREE_API int ddtree_verify_mla_plan(int batch, int n_nodes, int n_heads,
                           const int32_t* prefix_lens_host, int64_t pool_rows,
                           ddtree_plan_t* plan);

/* Same, for an explicit SM count and partial-kernel variant
 * (kernel = DDTREE_KERNEL_AUTO picks per shape).  num_sms >= 1 makes it a
 * pure host computation (used to plan off-GPU); num_sms = 0 asks the current
 * device, as ddtree_verify_mla_plan does: the SMs the chosen kernel's
 * clusters can occupy at once, which is below the SM count when a GPC's SMs
 * do not divide into whole clusters. */
DDTREE_API int ddtree_verify_mla_plan_ex(int batch, int n_nodes, int n_heads,
                              const int32_t* prefix_lens_host, int64_t pool_rows,
                              int num_sms, int kernel, ddtree_plan_t* plan);

/* Workspace bytes for a plan (a multiple of 256; the workspace must start
 * 256-byte aligned).  Returns 0 for a null plan. */
DDTREE_API size_t ddtree_verify_mla_workspace_size(const ddtree_plan_t* plan);

/*
 * Verify attention for ONE request (the single-request form).
 *   q_latent   [n_nodes, n_heads, 512] bf16, contiguous, 16-B aligned
 *   q_rope     [n_nodes, n_heads, 64]  bf16, contiguous, 16-B aligned
 *   kv_pool    [pool_rows, 576] bf16, row stride 576, 16-B aligned
 *   kv_indices [prefix_len + n_nodes] int32: prefix rows, then tree rows
 *              in node order (not bounds-checked against the pool here:
 *              use the batched form with a plan for that)
 *   tree_parent[n_nodes] int32 (device): -1 = root under the prefix end,
 *              else an earlier node
 *   out        [n_nodes, n_heads, 512] bf16 (written)
 *   lse        [n_nodes, n_heads] fp32, natural log (written)
 *   workspace  >= ddtree_verify_mla_workspace_size of the plan that
 *              ddtree_verify_mla_plan(1, n_nodes, n_heads, &prefix_len, ...)
 *              returns on this device
 * Plans internally on the host (no device calls besides the launches).
 */
DDTREE_API int ddtree_verify_mla(const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                      const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                      int prefix_len, const int32_t* tree_parent,
                      int n_nodes, int n_heads, float sm_scale,
                      ddtree_bf16_t* out, float* lse, void* workspace,
                      struct CUstream_st* stream);

/*
 * Verify attention for a batch under a plan.  Lengths are read on the
 * device, so one plan sized for the longest lengths can be captured once
 * and replayed with other indices and shorter prefixes.
 *   q_latent   [B*T, H, 512] bf16 (row stride plan->q_latent_row_stride)
 *   q_rope     [B*T, H, 64]  bf16 (row stride plan->q_rope_row_stride)
 *   kv_pool    [plan->pool_rows, 576] bf16
 *   kv_indices int32; request b owns kv_indices[kv_indptr[b] .. +P_b+T)
 *   kv_indptr  [B+1] int32 (device)
 *   prefix_lens[B] int32 (device), each <= the planned length
 *   tree_parent[B, T] int32 (device)
 *   out [B*T, H, 512] bf16, lse [B*T, H] fp32 (written)
 *   workspace of workspace_bytes >= plan->workspace_bytes, 256-B aligned
 */
DDTREE_API int ddtree_verify_mla_batched(const ddtree_plan_t* plan,
                              const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                              const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                              const int32_t* kv_indptr, const int32_t* prefix_lens,
                              const int32_t* tree_parent, float sm_scale,
                              ddtree_bf16_t* out, float* lse,
                              void* workspace, size_t workspace_bytes,
                              struct CUstream_st* stream);

/*
 * ddtree_verify_mla_batched with stage timing: records stage_events[0]
 * before the split-KV partial kernel, [1] between it and the combine
 * kernel, and [2] after the combine, all on `stream` (so the caller can time
 * each kernel with cudaEventElapsedTime, also inside a captured graph).
 * stage_events may be null, as may any of its three entries.
 */
DDTREE_API int ddtree_verify_mla_batched_timed(const ddtree_plan_t* plan,
                              const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                              const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                              const int32_t* kv_indptr, const int32_t* prefix_lens,
                              const int32_t* tree_parent, float sm_scale,
                              ddtree_bf16_t* out, float* lse,
                              void* workspace, size_t workspace_bytes,
                              struct CUstream_st* stream, struct CUevent_st* const* stage_events);

/*
 * Ancestor-mask stage on its own ("Chunk 66.1": the tree mask the host built
 * in 0.18 ms; here a device kernel).  anc_out[b*T + i] gets bit j set when
 * tree node j is i or one of i's ancestors.  Bad parents set
 * DDTREE_ST_BAD_PARENT in *status (device uint32, OR-ed; may be null) and
 * stop the walk at that node.
 */
DDTREE_API int ddtree_build_ancestor_mask(const int32_t* tree_parent, int batch, int n_nodes,
                               uint64_t* anc_out, uint32_t* status,
                               struct CUstream_st* stream);

/*
 * Read the device status word of the last call that used `workspace`
 * (synchronises `stream`).  *host_status gets the DDTREE_ST_* bits.  Returns
 * DDTREE_OK when the word is zero, DDTREE_EDEVICE_DATA otherwise.
 */
DDTREE_API int ddtree_verify_mla_check(const void* workspace, struct CUstream_st* stream,
                            uint32_t* host_status);

/*
 * Single-request verify attention that allocates nothing and needs no
 * workspace.  The pages have no counterpart of this entry point; it is an
 * addition for callers that cannot allocate device memory where they call
 * verify attention (an allocator that forbids raw cudaMalloc, a code path
 * where an allocation would synchronise the device, or a host integration
 * with nowhere to keep a workspace buffer).
 *
 * Arguments, layouts and results are those of ddtree_verify_mla without the
 * workspace.  The split-KV partials go to a scratch array built into the
 * library: DDTREE_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory that every
 * GPU loading the library keeps until the process exits.  When the usual
 * plan would need more scratch than that, the call uses fewer, longer KV
 * splits; a shape whose partials do not fit even with one split (more than
 * about 8,100 query rows, e.g. 64 nodes x 128 heads) returns
 * DDTREE_EWORKSPACE without launching anything.
 *  - The first call on each device looks up the scratch array's device
 *    address (cudaGetSymbolAddress, which can load the module); make that
 *    first call before any stream capture.
 *  - All calls on a device share the one scratch array, which keeps the
 *    previous call's contents; each call clears the status words it uses and
 *    writes every partial it reads.  Calls whose GPU work overlaps (other
 *    streams, other host threads) race on the array: serialise them.
 *  - The status word lives in the library's scratch, so neither device-data
 *    errors nor expired waits (DDTREE_ST_TIMEOUT) are observable through
 *    this entry point; indices are not checked against the pool size (as in
 *    ddtree_verify_mla).
 *  - The cached scratch address belongs to the device's context of the
 *    first call: do not use this entry point across a device reset
 *    (cudaDeviceReset) in the same process.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define DDTREE_NOALLOC_SCRATCH_BYTES (8u << 20)
DDTREE_API int ddtree_verify_mla_noalloc(const ddtree_bf16_t* q_latent, const ddtree_bf16_t* q_rope,
                              const ddtree_bf16_t* kv_pool, const int32_t* kv_indices,
                              int prefix_len, const int32_t* tree_parent,
                              int n_nodes, int n_heads, float sm_scale,
                              ddtree_bf16_t* out, float* lse, struct CUstream_st* stream);

/* Static text for a DDTREE_* return code. */
DDTREE_API const char* ddtree_status_str(int code);

#ifdef __cplusplus
}
#endif
#endif /* DDTREE_VERIFY_H */
