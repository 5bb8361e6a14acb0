// The C ABI declared in include/fa.h: argument validation, kernel choice,
// launch, status codes and the thread-local error text.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

thread_local std::string g_last_error;

fa_status fail(fa_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

fa_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t dtype_size(int dt) { return dt == FA_BF16 ? 2 : 4; }

fa_status validate(const fa::Problem &p)
{
    if (!p.q || !p.k || !p.v || !p.o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
    if (p.in_dtype != FA_BF16 && p.in_dtype != FA_FP32)
        return fail(FA_ERR_INVALID_ARG, "in_dtype %d is not an fa_dtype", p.in_dtype);
    if (p.o_dtype != FA_BF16 && p.o_dtype != FA_FP32)
        return fail(FA_ERR_INVALID_ARG, "o_dtype %d is not an fa_dtype", p.o_dtype);
    if (p.B < 1 || p.H < 1 || p.N < 1 || p.d < 1)
        return fail(FA_ERR_INVALID_ARG, "B, H, N, d must be >= 1 (got %lld, %lld, %lld, %lld)",
                    (long long)p.B, (long long)p.H, (long long)p.N, (long long)p.d);
    if (p.d > 1024) return fail(FA_ERR_UNSUPPORTED, "d = %lld exceeds the maximum head dimension 1024", (long long)p.d);
    if (p.B > (int64_t)INT32_MAX || p.H > (int64_t)INT32_MAX || p.N > (int64_t)INT32_MAX ||
        p.B * p.H > (int64_t)INT32_MAX / p.N)
        return fail(FA_ERR_UNSUPPORTED, "B * H * N must be below 2^31");
    if (!std::isfinite(p.scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    const size_t ei = dtype_size(p.in_dtype), eo = dtype_size(p.o_dtype);
    if (!aligned(p.q, ei) || !aligned(p.k, ei) || !aligned(p.v, ei) || !aligned(p.o, eo) ||
        (p.lse && !aligned(p.lse, 4)))
        return fail(FA_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    // O may not alias an input or LSE (the kernels read inputs after writing O rows).
    const size_t in_bytes = (size_t)(p.B * p.H * p.N * p.d) * ei;
    const size_t o_bytes = (size_t)(p.B * p.H * p.N * p.d) * eo;
    auto overlap = [](const void *a, size_t na, const void *b, size_t nb) {
        uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + nb && y < x + na;
    };
    if (overlap(p.o, o_bytes, p.q, in_bytes) || overlap(p.o, o_bytes, p.k, in_bytes) ||
        overlap(p.o, o_bytes, p.v, in_bytes) ||
        (p.lse && overlap(p.o, o_bytes, p.lse, (size_t)(p.B * p.H * p.N) * 4)))
        return fail(FA_ERR_INVALID_ARG, "o must not overlap q, k, v or lse");
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_forward_ex(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                        int64_t H, int64_t N, int64_t d, float scale, int causal, int in_dtype,
                        int o_dtype, void *stream, uint32_t flags)
{
    g_last_error.clear();
    fa::Problem p{q, k, v, o, lse, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
    fa_status st = validate(p);
    if (st != FA_OK) return st;
    if (flags & ~(uint32_t)FA_FLAG_GENERAL_PATH)
        return fail(FA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~(uint32_t)FA_FLAG_GENERAL_PATH);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!(flags & FA_FLAG_GENERAL_PATH) && fa::tc_supported(p)) {
        const char *detail = nullptr;
        e = fa::launch_tc(p, s, flags, &detail);
        if (e != cudaSuccess)
            return detail ? fail(FA_ERR_CUDA, "tensor-core launch: %s", detail) : cuda_fail(e, "tensor-core launch");
        return FA_OK;
    }
    e = fa::launch_general(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "general-d launch");
    return FA_OK;
}

fa_status fa_forward(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                     int64_t H, int64_t N, int64_t d, float scale, int causal, int in_dtype, int o_dtype,
                     void *stream)
{
    return fa_forward_ex(q, k, v, o, lse, B, H, N, d, scale, causal, in_dtype, o_dtype, stream, 0u);
}

fa_status fa_check_device_error(void *stream)
{
    g_last_error.clear();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t word = 0;
    e = fa::tc_take_error_word(&word, s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) return fail(FA_ERR_TIMEOUT, "a device pipeline wait gave up (error word 0x%x)", word);
    return FA_OK;
}

const char *fa_last_error(void) { return g_last_error.c_str(); }

const char *fa_version(void) { return "0.1.0 sm_103a"; }

}  // extern "C"
