// Batched (union-mask) sparse FFN on tensor cores -- placeholder until the
// mma kernel lands.
#include "internal.h"

namespace pi {

cudaError_t launch_sparse_union(int, int, const SparseParams &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pi
