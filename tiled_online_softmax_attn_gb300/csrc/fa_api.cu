// The C ABI declared in include/fa.h: argument validation, kernel choice,
// launch, status codes and the thread-local error text.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
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

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device-side copies of the tensors inside an fa_forward_host workspace.
struct HostLayout {
    size_t q, k, v, o, lse, total;
};

HostLayout host_layout(const fa::Problem &p)
{
    const size_t n = (size_t)(p.B * p.H * p.N * p.d);
    const size_t in_b = align256(n * dtype_size(p.in_dtype));
    const size_t o_b = align256(n * dtype_size(p.o_dtype));
    const size_t l_b = align256((size_t)(p.B * p.H * p.N) * 4);
    HostLayout L;
    L.q = 0;
    L.k = in_b;
    L.v = 2 * in_b;
    L.o = 3 * in_b;
    L.lse = 3 * in_b + o_b;
    L.total = 3 * in_b + o_b + l_b;
    return L;
}

// Streams and events the host-buffer pipeline uses, created once per device.
constexpr int MAX_DEVICES = 64;
constexpr int MAX_CHUNKS = 8;
struct PipelineRes {
    bool ready = false;
    cudaStream_t compute = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, copied[MAX_CHUNKS] = {}, computed[MAX_CHUNKS] = {};
};
PipelineRes g_pipes[MAX_DEVICES];
std::mutex g_pipes_mu;

cudaError_t pipeline_res(PipelineRes **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_pipes_mu);
    PipelineRes &r = g_pipes[dev];
    if (!r.ready) {
        const unsigned fl = cudaStreamNonBlocking;
        if ((e = cudaStreamCreateWithFlags(&r.compute, fl)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&r.d2h, fl)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&r.start, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int c = 0; c < MAX_CHUNKS; ++c) {
            if ((e = cudaEventCreateWithFlags(&r.copied[c], cudaEventDisableTiming)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&r.computed[c], cudaEventDisableTiming)) != cudaSuccess) return e;
        }
        r.ready = true;
    }
    *out = &r;
    return cudaSuccess;
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
    const uint32_t known = FA_FLAG_GENERAL_PATH | FA_FLAG_TEST_SKIP_KV_LOAD;
    if (flags & ~known) return fail(FA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~known);
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

size_t fa_host_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype)
{
    fa::Problem p{reinterpret_cast<const void *>(256), reinterpret_cast<const void *>(256),
                  reinterpret_cast<const void *>(256), reinterpret_cast<void *>(256), nullptr,
                  B, H, N, d, 1.0f, 0, in_dtype, o_dtype};
    std::string saved = g_last_error;
    // validate() also rejects the aliasing of these placeholder pointers, so
    // check the size and dtype rules alone
    bool ok = (in_dtype == FA_BF16 || in_dtype == FA_FP32) && (o_dtype == FA_BF16 || o_dtype == FA_FP32) &&
              B >= 1 && H >= 1 && N >= 1 && d >= 1 && d <= 1024 && B <= INT32_MAX && H <= INT32_MAX &&
              N <= INT32_MAX && B * H <= (int64_t)INT32_MAX / N;
    g_last_error = saved;
    return ok ? host_layout(p).total : 0;
}

fa_status fa_forward_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                          int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                          int in_dtype, int o_dtype, void *workspace, size_t workspace_bytes,
                          void *stream)
{
    g_last_error.clear();
    if (!q_h || !k_h || !v_h || !o_h) return fail(FA_ERR_INVALID_ARG, "q_h, k_h, v_h and o_h must be non-NULL");
    if (!workspace || !aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
    const size_t need = fa_host_workspace_size(B, H, N, d, in_dtype, o_dtype);
    if (need == 0) {
        // reuse fa_forward's messages for bad sizes and dtypes
        fa::Problem p{q_h, k_h, v_h, o_h, lse_h, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
        fa_status st = validate(p);
        return st != FA_OK ? st : fail(FA_ERR_INVALID_ARG, "bad problem size");
    }
    if (workspace_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "workspace of %zu bytes is below the %zu bytes needed", workspace_bytes, need);
    if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    fa::Problem full{q_h, k_h, v_h, o_h, lse_h, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
    const HostLayout L = host_layout(full);
    PipelineRes *res = nullptr;
    cudaError_t e = pipeline_res(&res);
    if (e != cudaSuccess) return cuda_fail(e, "creating the copy pipeline");
    cudaStream_t s_in = static_cast<cudaStream_t>(stream);

    const int64_t BH = B * H;
    const size_t ei = dtype_size(in_dtype), eo = dtype_size(o_dtype);
    const size_t head_elems = (size_t)(N * d);
    const size_t in_bytes_total = 3 * (size_t)BH * head_elems * ei;
    int chunks = (int)std::min<int64_t>({(int64_t)MAX_CHUNKS, BH, (int64_t)(in_bytes_total >> 22) + 1});
    chunks = std::max(chunks, 1);

    // the internal streams start after earlier work on the caller's stream
    if ((e = cudaEventRecord(res->start, s_in)) != cudaSuccess) return cuda_fail(e, "event record");
    if ((e = cudaStreamWaitEvent(res->compute, res->start, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
    if ((e = cudaStreamWaitEvent(res->d2h, res->start, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");

    for (int c = 0; c < chunks; ++c) {
        const int64_t h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks, nh = h1 - h0;
        if (nh == 0) continue;
        const size_t off_in = (size_t)h0 * head_elems * ei, n_in = (size_t)nh * head_elems * ei;
        const size_t off_o = (size_t)h0 * head_elems * eo, n_o = (size_t)nh * head_elems * eo;
        const size_t off_l = (size_t)h0 * N * 4, n_l = (size_t)nh * N * 4;
        const uint8_t *qh = static_cast<const uint8_t *>(q_h), *kh = static_cast<const uint8_t *>(k_h),
                      *vh = static_cast<const uint8_t *>(v_h);
        if ((e = cudaMemcpyAsync(ws + L.q + off_in, qh + off_in, n_in, cudaMemcpyHostToDevice, s_in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(ws + L.k + off_in, kh + off_in, n_in, cudaMemcpyHostToDevice, s_in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(ws + L.v + off_in, vh + off_in, n_in, cudaMemcpyHostToDevice, s_in)) != cudaSuccess ||
            (e = cudaEventRecord(res->copied[c], s_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(res->compute, res->copied[c], 0)) != cudaSuccess)
            return cuda_fail(e, "host-to-device copy");
        fa_status st = fa_forward(ws + L.q + off_in, ws + L.k + off_in, ws + L.v + off_in, ws + L.o + off_o,
                                  lse_h ? reinterpret_cast<float *>(ws + L.lse + off_l) : nullptr,
                                  1, nh, N, d, scale, causal, in_dtype, o_dtype, res->compute);
        if (st != FA_OK) return st;
        if ((e = cudaEventRecord(res->computed[c], res->compute)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(res->d2h, res->computed[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(static_cast<uint8_t *>(o_h) + off_o, ws + L.o + off_o, n_o,
                                 cudaMemcpyDeviceToHost, res->d2h)) != cudaSuccess)
            return cuda_fail(e, "device-to-host copy");
        if (lse_h && (e = cudaMemcpyAsync(reinterpret_cast<uint8_t *>(lse_h) + off_l, ws + L.lse + off_l, n_l,
                                          cudaMemcpyDeviceToHost, res->d2h)) != cudaSuccess)
            return cuda_fail(e, "device-to-host copy");
    }
    if ((e = cudaStreamSynchronize(res->d2h)) != cudaSuccess) return cuda_fail(e, "synchronize");
    if ((e = cudaStreamSynchronize(res->compute)) != cudaSuccess) return cuda_fail(e, "synchronize");
    return fa_check_device_error(stream);
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
