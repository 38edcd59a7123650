// Instantiates the launch layer for BF16 storage with pre as an input (one
// translation unit per storage type and coefficient source, so that the
// library's kernels compile in parallel).
#include "mhc_launch.cuh"

namespace mhc {
cudaError_t fwd_bf16(const FwdCall& c, const PlainCoeffs& k) { return fwd_dispatch<kBF16>(c, k); }
cudaError_t bwd_bf16(const BwdCall& c, const PlainCoeffs& k) { return bwd_dispatch<kBF16>(c, k); }
}  // namespace mhc
