/*
 * Reading a flattened custom attention mask back into the draft tree.
 *
 * Serving frameworks hand tree verify attention a boolean mask built on the
 * host ("Chunk 66.1", magik.net seg_66/chunk_1: the mask-build took 0.18 ms)
 * rather than a parent array.  The verify kernels here take the tree; this
 * call recovers it on the device: for request b the mask is a row-major
 * [T, P_b + T] byte array (nonzero = may attend) starting at element
 * mask_indptr[b] of custom_mask, row i for tree node i, column k < P_b for
 * prefix row k and column P_b + j for tree node j.  Because a node's
 * ancestors have smaller indices along its chain, the parent of node i is the
 * largest j < i that node i sees (-1 if none).
 *
 * The mask must be a tree mask: node i sees itself, every prefix row, and
 * exactly what its parent sees plus itself.  Anything else (a general DAG
 * mask, a hole in the prefix) sets DDTREE_ST_BAD_MASK; the parent rows are
 * still written by the rule above.  A mask span other than T*(P_b+T)
 * elements sets DDTREE_ST_BAD_LENGTH and that request's outputs are -1 / 0.
 *
 * Conventions as in ddtree_verify.h.
 */
#ifndef DDTREE_MASK_H_
#define DDTREE_MASK_H_

#include "ddtree_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes (multiple of 256, 256-byte aligned buffer): a 256-byte
 * status block (read with ddtree_verify_mla_check), one 64-bit row of mask
 * bits per node and a counter per request.  Cleared on the stream by every
 * call.  0 for sizes out of range. */
DDTREE_API size_t ddtree_tree_from_mask_workspace_size(int batch, int n_nodes);

/*
 *   custom_mask   bytes, the requests' [T, P_b+T] masks (device)
 *   mask_indptr   [batch+1] int64 element offsets (device)
 *   prefix_lens   [batch] int32 (device)
 *   tree_parent   [batch, n_nodes] int32 output (the verify layout)
 *   anc_bits      [batch, n_nodes] uint64 output, bit j = node j visible to
 *                 node i (the same bits ddtree_build_ancestor_mask gives), or
 *                 NULL
 * Errors: DDTREE_EINVAL (null/misaligned pointers, batch 1..1024, n_nodes
 * 1..64), DDTREE_EWORKSPACE, DDTREE_EUNSUPPORTED, DDTREE_ELAUNCH.
 */
DDTREE_API int ddtree_tree_from_mask(int batch, int n_nodes, const uint8_t* custom_mask, const int64_t* mask_indptr,
                                     const int32_t* prefix_lens, int32_t* tree_parent, uint64_t* anc_bits,
                                     void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_MASK_H_ */
