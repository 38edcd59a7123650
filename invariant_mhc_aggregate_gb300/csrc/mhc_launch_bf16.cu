// Instantiates the launch layer for BF16 storage (one translation unit per
// storage type so that the library's kernels compile in parallel).
#include "mhc_launch.cuh"

namespace mhc {
cudaError_t fwd_bf16(const FwdCall& c) { return fwd_dispatch<kBF16>(c); }
cudaError_t bwd_bf16(const BwdCall& c) { return bwd_dispatch<kBF16>(c); }
}  // namespace mhc
