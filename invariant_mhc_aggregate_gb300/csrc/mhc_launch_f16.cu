// Instantiates the launch layer for binary16 storage with pre as an input.
#include "mhc_launch.cuh"

namespace mhc {
cudaError_t fwd_f16(const FwdCall& c, const PlainCoeffs& k) { return fwd_dispatch<kF16>(c, k); }
cudaError_t bwd_f16(const BwdCall& c, const PlainCoeffs& k) { return bwd_dispatch<kF16>(c, k); }
}  // namespace mhc
