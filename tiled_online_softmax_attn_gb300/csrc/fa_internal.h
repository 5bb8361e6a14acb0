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

// Wide-head tensor-core path (fa_wide.cu): fp32 inputs with d % 128 == 0
// (d <= 1024), bf16 inputs with d % 128 == 0 and 256 <= d <= 1024.
struct WidePlan {
    bool ok;             // the path applies to this problem
    int nprod;           // 3: fp32 inputs as bf16 hi + lo pairs; 1: bf16 inputs
    int dv;              // width of the O slice a CTA owns (256 or 128)
    int n_q, n_kv, n_dv; // query tiles, key tiles, O slices
    int n_split, tiles_per_split;
    size_t off_split[6]; // workspace offsets of Q/K/V hi and lo copies (fp32 inputs)
    size_t off_opart, off_m, off_l, off_d;  // partial results when n_split > 1
    size_t workspace_bytes;
};
// max_splits = 1 plans a launch that needs no partials.
WidePlan wide_plan(const Problem &p, int max_splits);
cudaError_t launch_wide(const Problem &p, const WidePlan &w, void *workspace, cudaStream_t stream, uint32_t flags,
                        const char **detail);
cudaError_t wide_take_error_word(uint32_t *word, cudaStream_t stream);

// Sets the text fa_last_error returns on this host thread.
void set_last_error(const char *msg);

}  // namespace fa
