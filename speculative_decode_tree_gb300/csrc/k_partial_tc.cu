// Tensor-core (tcgen05 / TMEM) split-KV partial stage — placeholder until the
// kernel lands; plans never select it yet.
#include "common.cuh"

namespace ddtree {
cudaError_t launch_partial_tc(const VerifyArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ddtree
