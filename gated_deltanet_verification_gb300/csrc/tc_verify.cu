// Tensor-core (TMA + tcgen05) verification kernel.
#include "common.cuh"

namespace bole {

bool tc_verify_supported(const VerifyArgs &) { return false; }

cudaError_t launch_tc_verify(const VerifyArgs &, cudaStream_t) { return cudaErrorNotSupported; }

bool tc_commit_supported(const CommitArgs &) { return false; }

cudaError_t launch_tc_commit(const CommitArgs &, cudaStream_t) { return cudaErrorNotSupported; }

} // namespace bole
