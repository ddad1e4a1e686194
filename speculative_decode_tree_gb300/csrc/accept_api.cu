// Host side of the acceptance entry points (include/ddtree_accept.h):
// argument checks, workspace layout and the launch sequence.
#include <string.h>

#include "common.cuh"
#include "../../include/ddtree_accept.h"

namespace ddtree {
namespace {
constexpr size_t kStatusBytes = 256;
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline size_t keys_bytes(int batch, int n_nodes) {
  return ((size_t)batch * (n_nodes + 1) * 8 + 255) / 256 * 256;
}
inline size_t ticket_bytes(int batch) { return ((size_t)batch * 4 + 255) / 256 * 256; }
inline bool sizes_ok(int batch, int n_nodes) {
  return batch >= 1 && batch <= DDTREE_MAX_BATCH && n_nodes >= 1 && n_nodes <= DDTREE_MAX_NODES;
}
}  // namespace
}  // namespace ddtree

using namespace ddtree;

extern "C" size_t ddtree_accept_greedy_workspace_size(int batch, int n_nodes) {
  if (!sizes_ok(batch, n_nodes)) return 0;
  return kStatusBytes + keys_bytes(batch, n_nodes) + ticket_bytes(batch);
}

extern "C" int ddtree_accept_greedy(int batch, int n_nodes, int vocab, const ddtree_bf16_t* logits,
                                    const int32_t* draft_tokens, const int32_t* tree_parent,
                                    const int32_t* kv_indices, const int32_t* kv_indptr,
                                    const int32_t* prefix_lens, int32_t* accept_len, int32_t* next_token,
                                    int32_t* accepted_nodes, int32_t* commit_indices,
                                    int32_t* freed_indices, void* workspace, size_t workspace_bytes,
                                    struct CUstream_st* stream) {
  if (!sizes_ok(batch, n_nodes) || vocab < 1 || vocab > DDTREE_MAX_VOCAB) return DDTREE_EINVAL;
  const void* ptrs4[] = {draft_tokens, tree_parent, kv_indices, kv_indptr, prefix_lens, accept_len,
                         next_token, accepted_nodes, commit_indices, freed_indices};
  for (const void* p : ptrs4)
    if (!p || !aligned(p, 4)) return DDTREE_EINVAL;
  if (!logits || !aligned(logits, 2) || !workspace || !aligned(workspace, 256)) return DDTREE_EINVAL;
  if (workspace_bytes < ddtree_accept_greedy_workspace_size(batch, n_nodes)) return DDTREE_EWORKSPACE;
  DevInfo info;
  int rc = current_device_info(&info);
  if (rc != DDTREE_OK) return rc;
  if (info.major != 10 || info.minor != 3) return DDTREE_EUNSUPPORTED;

  AcceptArgs a;
  memset(&a, 0, sizeof(a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.logits = logits;
  a.draft = draft_tokens;
  a.parent = tree_parent;
  a.kv_indices = kv_indices;
  a.kv_indptr = kv_indptr;
  a.prefix_lens = prefix_lens;
  a.keys = reinterpret_cast<uint64_t*>(ws + kStatusBytes);
  a.tickets = reinterpret_cast<uint32_t*>(ws + kStatusBytes + keys_bytes(batch, n_nodes));
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.accepted_nodes = accepted_nodes;
  a.commit_indices = commit_indices;
  a.freed_indices = freed_indices;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.batch = batch;
  a.n_nodes = n_nodes;
  a.vocab = vocab;
  a.num_sms = info.sms;
  cudaStream_t s = (cudaStream_t)stream;
  // Status word, argmax keys and tickets start at zero (a key of 0 is below
  // every real value's key).  The workspace keeps nothing between calls.
  if (cudaMemsetAsync(ws, 0, ddtree_accept_greedy_workspace_size(batch, n_nodes), s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ECUDA;
  }
  if (launch_accept(a, s) != cudaSuccess) {
    cudaGetLastError();
    return DDTREE_ELAUNCH;
  }
  return DDTREE_OK;
}
