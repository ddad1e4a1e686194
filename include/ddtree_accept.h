/*
 * Greedy acceptance of a verified DDTree draft tree and the KV commit that
 * follows it: the step right after verify attention in a speculative decode
 * loop ("Chunk 66.0", magik.net seg_66/chunk_0: the DDTree commit length --
 * 7-8 tokens per step on predictable text -- is what this step produces).
 *
 * The verify forward scores every tree node; the target model's token at a
 * position is the argmax of its logits (first index among equal maxima).
 * Starting at the prefix end, the walk accepts the child whose drafted token
 * equals the target's token (the smallest node index if several do), moves
 * to it and repeats; it stops when no child matches.  The target's token
 * after the last accepted node is the extra token every step commits.  The
 * KV rows of the accepted nodes become committed context, in path order; the
 * rows of the other nodes are released.
 *
 * Same conventions as ddtree_verify.h: caller-owned device buffers, no
 * allocation, everything enqueued on `stream`, no host synchronisation.
 */
#ifndef DDTREE_ACCEPT_H_
#define DDTREE_ACCEPT_H_

#include "ddtree_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DDTREE_MAX_VOCAB (1 << 26)

/* Workspace bytes for `batch` requests of `n_nodes` nodes (a multiple of 256;
 * the workspace must be 256-byte aligned).  Layout: a 256-byte status block
 * (same status bits as verify: read it with ddtree_verify_mla_check), one
 * 64-bit argmax key per scored row, one 32-bit counter per request.  Every
 * call clears it on the stream first; it carries nothing between calls.
 * 0 for sizes out of range. */
DDTREE_API size_t ddtree_accept_greedy_workspace_size(int batch, int n_nodes);

/*
 * Greedy acceptance + commit for `batch` requests.
 *   logits          [batch, n_nodes+1, vocab] bf16, contiguous.  Row 0 of a
 *                   request is the target's prediction at the end of its
 *                   prefix (it scores the roots, parent = -1); row 1+i the
 *                   prediction after tree node i.
 *   draft_tokens    [batch, n_nodes] int32: the drafted token of each node
 *   tree_parent     [batch, n_nodes] int32: -1 or an earlier node
 *   kv_indices      int32, per request: prefix_lens[b] prefix rows, then the
 *                   n_nodes tree rows in node order (the verify layout)
 *   kv_indptr       [batch+1] int32, prefix_lens [batch] int32 (device)
 * Outputs (device, caller-owned, fully written):
 *   accept_len      [batch] int32: accepted tree nodes (the commit length is
 *                   accept_len + 1 with the extra token)
 *   next_token      [batch] int32: the target's token after the accepted path
 *   accepted_nodes  [batch, n_nodes] int32: path in order, then -1
 *   commit_indices  [batch, n_nodes] int32: pool rows of the accepted nodes in
 *                   path order, then -1
 *   freed_indices   [batch, n_nodes] int32: pool rows of the other nodes in
 *                   node order, then -1
 * Device-data errors set status bits instead of faulting: BAD_PARENT (a
 * parent not in [-1, i)), BAD_LENGTH (kv_indptr span != prefix + n_nodes;
 * that request's row outputs are then -1).
 * Errors: DDTREE_EINVAL (null or misaligned pointer, sizes out of range:
 * batch 1..1024, n_nodes 1..64, vocab 1..2^26), DDTREE_EWORKSPACE,
 * DDTREE_EUNSUPPORTED (no sm_103 device current), DDTREE_ELAUNCH.
 */
DDTREE_API int ddtree_accept_greedy(int batch, int n_nodes, int vocab, const ddtree_bf16_t* logits,
                                    const int32_t* draft_tokens, const int32_t* tree_parent,
                                    const int32_t* kv_indices, const int32_t* kv_indptr,
                                    const int32_t* prefix_lens, int32_t* accept_len, int32_t* next_token,
                                    int32_t* accepted_nodes, int32_t* commit_indices,
                                    int32_t* freed_indices, void* workspace, size_t workspace_bytes,
                                    struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_ACCEPT_H_ */
