// Tensor-core attention forward (tcgen05 + TMA) -- placeholder until the
// kernel lands: reports itself unsupported so the general path runs.
#include <cuda_runtime.h>
#include <cstdint>
#include "fa_internal.h"

namespace fa {

__device__ uint32_t g_tc_error_word;

bool tc_supported(const Problem &) { return false; }

cudaError_t launch_tc(const Problem &, cudaStream_t, uint32_t, const char **detail)
{
    *detail = "tensor-core kernel not built";
    return cudaErrorNotSupported;
}

cudaError_t tc_take_error_word(uint32_t *word, cudaStream_t stream)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_tc_error_word, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || *word == 0) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tc_error_word, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace fa
