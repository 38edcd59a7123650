/* A plain C program using the library through its C ABI only (no Python, no
 * PyTorch): it reads residual / pre / g from files, allocates device memory
 * with the CUDA runtime, runs the forward and the backward on a stream of its
 * own, and writes out / grad_residual / grad_pre to files.
 *
 *   c_consumer <dir> <T> <H>
 *   reads  dir/residual.bin (BF16 [T,4,H]), dir/pre.bin (FP32 [T,4]), dir/g.bin (BF16 [T,H])
 *   writes dir/out.bin, dir/grad_residual.bin, dir/grad_pre.bin
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mhc_h_aggregate.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    void* p = malloc(bytes);
    size_t got = p ? fread(p, 1, bytes, f) : 0;
    fclose(f);
    if (got != bytes) {
        free(p);
        return NULL;
    }
    return p;
}

static int write_file(const char* dir, const char* name, const void* p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    size_t put = fwrite(p, 1, bytes, f);
    fclose(f);
    return put != bytes;
}

#define CHECK_CUDA(x)                                                                   \
    do {                                                                                \
        cudaError_t e_ = (x);                                                           \
        if (e_ != cudaSuccess) {                                                        \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));             \
            return 2;                                                                   \
        }                                                                               \
    } while (0)

#define CHECK_MHC(x)                                                                    \
    do {                                                                                \
        mhc_status_t s_ = (x);                                                          \
        if (s_ != MHC_OK) {                                                             \
            fprintf(stderr, "%s failed: %s\n", #x, mhc_status_string(s_));              \
            return 3;                                                                   \
        }                                                                               \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 4) {
        fprintf(stderr, "usage: %s <dir> <T> <H>\n", argv[0]);
        return 1;
    }
    const char* dir = argv[1];
    const int64_t T = atoll(argv[2]), H = atoll(argv[3]);
    const size_t rb = (size_t)T * 4 * (size_t)H * 2, pb = (size_t)T * 16, gb = (size_t)T * (size_t)H * 2;
    void* h_res = read_file(dir, "residual.bin", rb);
    void* h_pre = read_file(dir, "pre.bin", pb);
    void* h_g = read_file(dir, "g.bin", gb);
    if (!h_res || !h_pre || !h_g) {
        fprintf(stderr, "cannot read inputs\n");
        return 1;
    }
    if (mhc_h_aggregate_abi_version() < 1) return 4;

    void *d_res, *d_pre, *d_g, *d_out, *d_gr, *d_gp;
    CHECK_CUDA(cudaMalloc(&d_res, rb));
    CHECK_CUDA(cudaMalloc(&d_pre, pb));
    CHECK_CUDA(cudaMalloc(&d_g, gb));
    CHECK_CUDA(cudaMalloc(&d_out, gb));
    CHECK_CUDA(cudaMalloc(&d_gr, rb));
    CHECK_CUDA(cudaMalloc(&d_gp, pb));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    CHECK_CUDA(cudaMemcpyAsync(d_res, h_res, rb, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_pre, h_pre, pb, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_g, h_g, gb, cudaMemcpyHostToDevice, stream));

    /* a rejected call launches nothing and says why */
    if (mhc_h_aggregate_fwd(d_res, (const float*)d_pre, d_res, T, H, (mhc_stream_t)stream) !=
        MHC_ERR_INVALID_ARG) {
        fprintf(stderr, "overlapping output was not rejected\n");
        return 5;
    }
    CHECK_MHC(mhc_h_aggregate_fwd(d_res, (const float*)d_pre, d_out, T, H, (mhc_stream_t)stream));
    CHECK_MHC(mhc_h_aggregate_bwd(d_g, d_res, (const float*)d_pre, d_gr, (float*)d_gp, T, H,
                                  (mhc_stream_t)stream));

    void* h_out = malloc(gb);
    void* h_gr = malloc(rb);
    void* h_gp = malloc(pb);
    CHECK_CUDA(cudaMemcpyAsync(h_out, d_out, gb, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(h_gr, d_gr, rb, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(h_gp, d_gp, pb, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    if (write_file(dir, "out.bin", h_out, gb) || write_file(dir, "grad_residual.bin", h_gr, rb) ||
        write_file(dir, "grad_pre.bin", h_gp, pb)) {
        fprintf(stderr, "cannot write outputs\n");
        return 1;
    }
    printf("ok T=%lld H=%lld\n", (long long)T, (long long)H);
    return 0;
}
