// Instantiates the launch layer for IEEE binary16 storage (one translation
// unit per storage type so that the library's kernels compile in parallel).
#include "mhc_launch.cuh"

namespace mhc {
cudaError_t fwd_f16(const FwdCall& c) { return fwd_dispatch<kF16>(c); }
cudaError_t bwd_f16(const BwdCall& c) { return bwd_dispatch<kF16>(c); }
}  // namespace mhc
