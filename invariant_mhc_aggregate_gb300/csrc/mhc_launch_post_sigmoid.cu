// Launches the mHC post kernels with post computed from the mix
// (SigmoidCoeffs), for both storage types.
#include "mhc_launch_post.cuh"

namespace mhc {

cudaError_t post_fwd(const PostFwdCall& c, const SigmoidCoeffs& k, int dtype) {
    return post_launch::fwd(c, k, dtype);
}

cudaError_t post_bwd(const PostBwdCall& c, const SigmoidCoeffs& k, int dtype) {
    return post_launch::bwd(c, k, dtype);
}

}  // namespace mhc
