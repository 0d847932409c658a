// Prefill over row-indexed lists (placeholder until the tensor-core kernel lands).
#include "fa_internal.cuh"

namespace far {
bool prefill_supported(int D, int kind) { (void)D; (void)kind; return false; }
cudaError_t prefill_launch(const PrefillParams& p, cudaStream_t st) { (void)p; (void)st; return cudaErrorNotSupported; }
}  // namespace far
