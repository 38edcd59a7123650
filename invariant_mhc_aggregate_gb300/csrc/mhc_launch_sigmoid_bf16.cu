// Instantiates the launch layer for BF16 storage with pre computed in the
// kernels from the mix (sigmoid of alpha * mix + b).
#include "mhc_launch.cuh"

namespace mhc {
cudaError_t fwd_bf16(const FwdCall& c, const SigmoidCoeffs& k) { return fwd_dispatch<kBF16>(c, k); }
cudaError_t bwd_bf16(const BwdCall& c, const SigmoidCoeffs& k) { return bwd_dispatch<kBF16>(c, k); }
}  // namespace mhc
