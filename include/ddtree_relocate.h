/*
 * Tier-1 KV relocation ("Chunk 66.1", magik.net seg_66/chunk_1: Tier 0 kept a
 * request's KV contiguous through the allocator; Tier 1, live relocation of
 * rows already scattered over a churned token-granular pool, was deferred).
 *
 * For each request b with pool rows idx_b[0..n_b) (its slice of kv_indices,
 * n_b = kv_indptr[b+1] - kv_indptr[b]) and a destination start d_b chosen by
 * the caller's allocator, the call copies pool[idx_b[k]] to pool[d_b + k] and
 * rewrites idx_b[k] = d_b + k, so the request then takes the contiguous path
 * of verify attention.  The old row numbers are written to old_indices (if
 * given) for the allocator to release.
 *
 * All or nothing: before anything moves, the call checks on the device that
 * every index lies in the pool (else DDTREE_ST_BAD_INDEX), every destination
 * region lies in the pool and kv_indptr is consistent with total_rows (else
 * DDTREE_ST_BAD_LENGTH), and no destination row is in two regions or holds a
 * row the batch reads (else DDTREE_ST_OVERLAP).  If any bit is set the pool
 * and the indices are left as they were (old_indices still receives a copy of
 * the indices).  Read the bits with ddtree_verify_mla_check(workspace, ...).
 *
 * Conventions as in ddtree_verify.h: caller-owned device buffers, no
 * allocation, everything on `stream`, no host synchronisation.
 */
#ifndef DDTREE_RELOCATE_H_
#define DDTREE_RELOCATE_H_

#include "ddtree_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes for a pool of `pool_rows` rows: a 256-byte status block and
 * a bitmap with one bit per pool row (rounded to 256 bytes).  The call clears
 * it on the stream first.  0 when pool_rows is out of range (1 .. 2^31-1). */
DDTREE_API size_t ddtree_relocate_kv_workspace_size(int64_t pool_rows);

/*
 *   batch        number of requests (1 .. 1024)
 *   total_rows   host copy of kv_indptr[batch] (sizes the grid; a device value
 *                that differs sets BAD_LENGTH)
 *   kv_pool      [pool_rows, 576] bf16, 16-byte aligned; updated in place
 *   kv_indices   [total_rows] int32, updated in place
 *   kv_indptr    [batch+1] int32 (device), dest_base [batch] int32 (device)
 *   old_indices  [total_rows] int32 output, or NULL
 * Errors: DDTREE_EINVAL (null/misaligned pointers, sizes out of range),
 * DDTREE_EWORKSPACE, DDTREE_EUNSUPPORTED, DDTREE_ELAUNCH.
 */
DDTREE_API int ddtree_relocate_kv(int batch, int64_t total_rows, ddtree_bf16_t* kv_pool, int64_t pool_rows,
                                  int32_t* kv_indices, const int32_t* kv_indptr, const int32_t* dest_base,
                                  int32_t* old_indices, void* workspace, size_t workspace_bytes,
                                  struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_RELOCATE_H_ */
