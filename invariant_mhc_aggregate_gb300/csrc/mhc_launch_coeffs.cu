// Launches the coefficient kernels of their own: pre = sigmoid(alpha * mix + b)
// and the reduction of the gradients of alpha and b over tokens.
#include "mhc_launch.cuh"

namespace mhc {

template <int N>
static cudaError_t pre_sigmoid_n(const float* mix, const float* alpha, const float* b, float* pre,
                                 uint64_t T, int num_sms, cudaStream_t stream) {
    const uint64_t count = T * uint64_t(N);
    const uint32_t blocks = grid_for(count, kCoeffBlock, uint64_t(num_sms) * 8);
    return launch(pre_sigmoid_kernel<N>, blocks, kCoeffBlock, stream, mix, alpha, b, pre, count);
}

cudaError_t pre_sigmoid(const float* mix, const float* alpha, const float* b, float* pre,
                        uint64_t T, int n, int num_sms, cudaStream_t stream) {
    switch (n) {
        case 1: return pre_sigmoid_n<1>(mix, alpha, b, pre, T, num_sms, stream);
        case 2: return pre_sigmoid_n<2>(mix, alpha, b, pre, T, num_sms, stream);
        case 4: return pre_sigmoid_n<4>(mix, alpha, b, pre, T, num_sms, stream);
        default: return pre_sigmoid_n<8>(mix, alpha, b, pre, T, num_sms, stream);
    }
}

// One cluster of 8 CTAs (see sigmoid_param_grad_kernel), with programmatic
// stream serialization like every launch here.
template <int N>
static cudaError_t param_grad_n(const float* grad_z, const float* mix, float* grad_b,
                                float* grad_alpha, uint64_t T, bool vec, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kParamClusterCtas);
    cfg.blockDim = dim3(kParamThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kParamClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sigmoid_param_grad_kernel<N>, grad_z, mix, grad_b, grad_alpha,
                              T, vec);
}

cudaError_t sigmoid_param_grad(const float* grad_z, const float* mix, float* grad_b,
                               float* grad_alpha, uint64_t T, int n, bool vec, cudaStream_t stream) {
    switch (n) {
        case 1: return param_grad_n<1>(grad_z, mix, grad_b, grad_alpha, T, vec, stream);
        case 2: return param_grad_n<2>(grad_z, mix, grad_b, grad_alpha, T, vec, stream);
        case 4: return param_grad_n<4>(grad_z, mix, grad_b, grad_alpha, T, vec, stream);
        default: return param_grad_n<8>(grad_z, mix, grad_b, grad_alpha, T, vec, stream);
    }
}

}  // namespace mhc
