// Internal interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

// One forward problem, already validated by the C ABI.
struct Problem {
    const void *q, *k, *v;
    void *o;
    float *lse;            // may be null
    int64_t B, H, N, d;
    float scale;
    int causal;
    int in_dtype;          // fa_dtype
    int o_dtype;           // fa_dtype
};

// General-d CUDA-core kernel (any d <= 1024, bf16 or fp32 in and out).
cudaError_t launch_general(const Problem &p, cudaStream_t stream);

// Tensor-core kernel (tcgen05 + TMA): bf16 in, d in {64, 128}.
bool tc_supported(const Problem &p);
// Returns cudaSuccess or an error; *detail receives a static description on
// failures that are not CUDA errors (tensor-map encoding).
cudaError_t launch_tc(const Problem &p, cudaStream_t stream, uint32_t flags, const char **detail);

// Reads and clears the device error word of the tensor-core kernel.
cudaError_t tc_take_error_word(uint32_t *word, cudaStream_t stream);

}  // namespace fa
