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

// Text and status of the last failure on this host thread; every entry
// point that can fail clears both first.
thread_local std::string g_last_error;
thread_local fa_status g_last_status = FA_OK;

void clear_error()
{
    g_last_error.clear();
    g_last_status = FA_OK;
}

fa_status fail(fa_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    g_last_status = s;
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

// The size and dtype rules of validate(), without pointers.
bool size_ok(const fa::Problem &p)
{
    return (p.in_dtype == FA_BF16 || p.in_dtype == FA_FP32) && (p.o_dtype == FA_BF16 || p.o_dtype == FA_FP32) &&
           p.B >= 1 && p.H >= 1 && p.N >= 1 && p.d >= 1 && p.d <= 1024 && p.B <= INT32_MAX && p.H <= INT32_MAX &&
           p.N <= INT32_MAX && p.B * p.H <= (int64_t)INT32_MAX / p.N;
}

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
// One call uses them at a time: `in_use` is held for the whole (synchronous)
// call, so concurrent callers on one device take turns instead of interleaving
// their event records and waits on the same streams.
constexpr int MAX_DEVICES = 64;
constexpr int MAX_CHUNKS = 8;
struct PipelineRes {
    bool ready = false;
    cudaStream_t compute = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, copied[MAX_CHUNKS] = {}, computed[MAX_CHUNKS] = {};
    std::mutex in_use;
};
PipelineRes g_pipes[MAX_DEVICES];
std::mutex g_pipes_mu;

cudaError_t pipeline_res(PipelineRes **out, std::unique_lock<std::mutex> *hold)
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
    *hold = std::unique_lock<std::mutex>(r.in_use);
    *out = &r;
    return cudaSuccess;
}

// Byte range [lo, hi) a strided tensor can touch.
struct Extent {
    uintptr_t lo, hi;
};

Extent extent_of(const void *ptr, const int64_t st[3], const int64_t size[3], int64_t width, size_t elt)
{
    int64_t last = width - 1;
    for (int i = 0; i < 3; ++i) last += (size[i] - 1) * st[i];
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    return {lo, lo + (uintptr_t)(last + 1) * elt};
}

// No two elements of a strided tensor share an address: with the dimensions
// sorted by stride, each stride exceeds the span of the smaller ones.
bool no_self_overlap(const int64_t st[3], const int64_t size[3], int64_t width)
{
    struct D {
        int64_t stride, size;
    } dd[4] = {{1, width}, {st[0], size[0]}, {st[1], size[1]}, {st[2], size[2]}};
    for (int i = 1; i < 4; ++i)
        for (int j = i; j > 0 && dd[j].stride < dd[j - 1].stride; --j) {
            D t = dd[j];
            dd[j] = dd[j - 1];
            dd[j - 1] = t;
        }
    int64_t span = 0;  // largest offset reachable with the dimensions so far
    for (int i = 0; i < 4; ++i) {
        if (dd[i].size <= 1) continue;
        if (dd[i].stride <= span) return false;
        span += (dd[i].size - 1) * dd[i].stride;
    }
    return true;
}

fa_status validate_general(const fa::Problem &p)
{
    if (!p.q || !p.k || !p.v || !p.o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
    if (p.in_dtype != FA_BF16 && p.in_dtype != FA_FP32)
        return fail(FA_ERR_INVALID_ARG, "in_dtype %d is not an fa_dtype", p.in_dtype);
    if (p.o_dtype != FA_BF16 && p.o_dtype != FA_FP32)
        return fail(FA_ERR_INVALID_ARG, "o_dtype %d is not an fa_dtype", p.o_dtype);
    const int64_t Nk = p.Nk, dv = p.dv;
    if (p.B < 1 || p.H < 1 || p.N < 1 || Nk < 1 || p.d < 1 || dv < 1)
        return fail(FA_ERR_INVALID_ARG, "B, H, Nq, Nk, dk, dv must be >= 1");
    if (p.d > 1024 || dv > 1024) return fail(FA_ERR_UNSUPPORTED, "dk and dv must be <= 1024");
    const int64_t nmax = std::max(p.N, Nk);
    if (p.B > (int64_t)INT32_MAX || p.H > (int64_t)INT32_MAX || nmax > (int64_t)INT32_MAX ||
        p.B * p.H > (int64_t)INT32_MAX / nmax)
        return fail(FA_ERR_UNSUPPORTED, "B * H * max(Nq, Nk) must be below 2^31");
    if (!std::isfinite(p.scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    const size_t ei = dtype_size(p.in_dtype), eo = dtype_size(p.o_dtype);
    if (!aligned(p.q, ei) || !aligned(p.k, ei) || !aligned(p.v, ei) || !aligned(p.o, eo) ||
        (p.lse && !aligned(p.lse, 4)))
        return fail(FA_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    int64_t st[4][3];
    for (int t = 0; t < 4; ++t) {
        fa::strides_of(p, t, st[t]);
        for (int i = 0; i < 3; ++i)
            if (st[t][i] < 0) return fail(FA_ERR_INVALID_ARG, "strides must be >= 0");
    }
    const int64_t sq[3] = {p.B, p.H, p.N}, sk[3] = {p.B, p.H, Nk};
    if (!no_self_overlap(st[3], sq, dv)) return fail(FA_ERR_INVALID_ARG, "o's strides make its elements overlap");
    const Extent eo_ = extent_of(p.o, st[3], sq, dv, eo);
    const Extent ins[3] = {extent_of(p.q, st[0], sq, p.d, ei), extent_of(p.k, st[1], sk, p.d, ei),
                           extent_of(p.v, st[2], sk, dv, ei)};
    for (const Extent &x : ins)
        if (eo_.lo < x.hi && x.lo < eo_.hi) return fail(FA_ERR_INVALID_ARG, "o must not overlap q, k or v");
    if (p.lse) {
        const uintptr_t l0 = reinterpret_cast<uintptr_t>(p.lse), l1 = l0 + (uintptr_t)(p.B * p.H * p.N) * 4;
        if (eo_.lo < l1 && l0 < eo_.hi) return fail(FA_ERR_INVALID_ARG, "o must not overlap lse");
    }
    return FA_OK;
}

// The error words of the three kernel families, read with one synchronisation
// of the stream (after the work already queued on it) into pinned memory of
// this host thread, and cleared where set.
cudaError_t take_error_words(uint32_t *word, cudaStream_t s)
{
    constexpr int NW = 4;
    thread_local uint32_t *host = nullptr;  // pinned, NW words, one block per host thread
    if (!host) {
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void **>(&host), NW * sizeof(uint32_t), cudaHostAllocDefault);
        if (e != cudaSuccess) return e;
    }
    uint32_t *dev[NW] = {nullptr, nullptr, nullptr, nullptr};
    cudaError_t e = fa::tc_error_word_ptr(&dev[0]);
    if (e == cudaSuccess) e = fa::wide_error_word_ptr(&dev[1]);
    if (e == cudaSuccess) e = fa::bwd_error_word_ptr(&dev[2]);
    if (e == cudaSuccess) e = fa::bwdw_error_word_ptr(&dev[3]);
    for (int i = 0; i < NW && e == cudaSuccess; ++i)
        e = cudaMemcpyAsync(&host[i], dev[i], sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *word = host[0] | host[1] | host[2] | host[3];
    if (*word == 0) return cudaSuccess;
    for (int i = 0; i < NW && e == cudaSuccess; ++i)
        if (host[i]) e = cudaMemsetAsync(dev[i], 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

// Heads per pipelined chunk of fa_forward_host: up to MAX_CHUNKS chunks of
// at least ~4 MB of input each.
int host_chunks(const fa::Problem &p)
{
    const int64_t BH = p.B * p.H;
    const size_t in_bytes_total = 3 * (size_t)(BH * p.N * p.d) * dtype_size(p.in_dtype);
    const int chunks = (int)std::min<int64_t>({(int64_t)MAX_CHUNKS, BH, (int64_t)(in_bytes_total >> 22) + 1});
    return std::max(chunks, 1);
}

// First head of chunk c of fa_forward_host.  Chunk sizes fall linearly
// (boundaries at BH (1 - (1 - c / K)^2)): the copies in are the bottleneck and
// the kernel and the copy out of the last chunk are the only work not hidden
// behind them, so the last chunk is the smallest.
int64_t chunk_head(int64_t BH, int chunks, int c)
{
    if (c >= chunks) return BH;
    const double r = 1.0 - (double)c / chunks;
    return std::min<int64_t>(BH, (int64_t)std::llround((double)BH * (1.0 - r * r)));
}

// Kernel workspace for one chunk of fa_forward_host (the largest chunk).
size_t chunk_workspace(const fa::Problem &p)
{
    const int64_t BH = p.B * p.H;
    const int chunks = host_chunks(p);
    int64_t largest = 1;
    for (int c = 0; c < chunks; ++c)
        largest = std::max(largest, chunk_head(BH, chunks, c + 1) - chunk_head(BH, chunks, c));
    fa::Problem c = p;
    c.B = 1;
    c.H = largest;
    if (fa::tc_supported(c)) return 0;
    const fa::WidePlan w = fa::wide_plan(c, 1 << 20);
    return w.ok ? w.workspace_bytes : 0;
}

// Kernel choice shared by every entry point: the 64/128 tensor-core kernel,
// then the wide-head tensor-core path (within the workspace given), then the
// general CUDA-core kernel.
fa_status dispatch(const fa::Problem &p, void *workspace, size_t workspace_bytes, cudaStream_t s, uint32_t flags)
{
    const uint32_t known = FA_FLAG_GENERAL_PATH | FA_FLAG_TEST_SKIP_KV_LOAD;
    if (flags & ~known) return fail(FA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~known);
    if (workspace && !aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    cudaError_t e;
    const char *detail = nullptr;
    if (!(flags & FA_FLAG_GENERAL_PATH)) {
        if (fa::tc_supported(p)) {
            // with a workspace, too few work items are spread over key-range splits
            const fa::TcSplit sp = (workspace && !flags) ? fa::tc_split_plan(p) : fa::TcSplit{1, 0, 0};
            if (sp.n_split > 1 && workspace_bytes >= sp.workspace_bytes)
                e = fa::launch_tc_split(p, sp, workspace, s, &detail);
            else
                e = fa::launch_tc(p, s, flags, &detail);
            if (e != cudaSuccess)
                return detail ? fail(FA_ERR_CUDA, "tensor-core launch: %s", detail) : cuda_fail(e, "tensor-core launch");
            return FA_OK;
        }
        fa::WidePlan w = fa::wide_plan(p, workspace ? 1 << 20 : 1);
        if (w.ok && workspace && workspace_bytes < w.workspace_bytes) w = fa::wide_plan(p, 1);
        if (w.ok && (w.workspace_bytes == 0 || (workspace && workspace_bytes >= w.workspace_bytes))) {
            e = fa::launch_wide(p, w, workspace, s, flags, &detail);
            if (e != cudaSuccess)
                return detail ? fail(FA_ERR_CUDA, "wide-head launch: %s", detail) : cuda_fail(e, "wide-head launch");
            return FA_OK;
        }
    }
    e = fa::launch_general(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "general-d launch");
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype, int causal)
{
    const uintptr_t a = 256;  // placeholder, aligned pointers for planning only
    fa::Problem p{reinterpret_cast<const void *>(a), reinterpret_cast<const void *>(a), reinterpret_cast<const void *>(a),
                  reinterpret_cast<void *>(a), nullptr, B, H, N, d, 1.0f, causal != 0, in_dtype, o_dtype};
    if (!size_ok(p)) return 0;
    if (fa::tc_supported(p)) return fa::tc_split_plan(p).workspace_bytes;
    const fa::WidePlan w = fa::wide_plan(p, 1 << 20);
    return w.ok ? w.workspace_bytes : 0;
}

int fa_plan(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype, int causal,
            size_t workspace_bytes, char *desc, size_t desc_len)
{
    const uintptr_t a = 256;
    fa::Problem p{reinterpret_cast<const void *>(a), reinterpret_cast<const void *>(a), reinterpret_cast<const void *>(a),
                  reinterpret_cast<void *>(a), nullptr, B, H, N, d, 1.0f, causal != 0, in_dtype, o_dtype};
    if (!size_ok(p)) return -1;
    char buf[160];
    int launches;
    if (fa::tc_supported(p)) {
        const fa::TcSplit sp = fa::tc_split_plan(p);
        const char *rows = fa::tc_item_rows(p) == 128 ? ", one query tile per item" : "";
        if (sp.n_split > 1 && workspace_bytes >= sp.workspace_bytes) {
            launches = 2;
            snprintf(buf, sizeof(buf), "tensor-core d=%lld key splits=%d%s", (long long)d, sp.n_split, rows);
        } else {
            launches = 1;
            snprintf(buf, sizeof(buf), "tensor-core d=%lld%s", (long long)d, rows);
        }
    } else {
        fa::WidePlan w = fa::wide_plan(p, workspace_bytes ? 1 << 20 : 1);
        if (w.ok && workspace_bytes && workspace_bytes < w.workspace_bytes) w = fa::wide_plan(p, 1);
        if (w.ok && (w.workspace_bytes == 0 || workspace_bytes >= w.workspace_bytes)) {
            launches = (w.nprod == 3 ? 1 : 0) + 1 + (w.n_split > 1 ? 1 : 0);
            snprintf(buf, sizeof(buf), "wide-head %s dv=%d splits=%d cluster=%d",
                     w.nprod == 3 ? "fp32 as bf16 hi+lo" : "bf16", w.dv, w.n_split, w.cluster);
        } else {
            launches = 1;
            snprintf(buf, sizeof(buf), "general-d");
        }
    }
    if (desc && desc_len) snprintf(desc, desc_len, "%s", buf);
    return launches;
}

namespace {
fa::Problem problem_of(const fa_params *a)
{
    fa::Problem p{a->q, a->k, a->v, a->o, a->lse, a->B, a->H, a->Nq, a->dk, a->scale, a->causal != 0,
                  a->in_dtype, a->o_dtype};
    p.Nk = a->Nk;
    p.dv = a->dv;
    for (int i = 0; i < 3; ++i) {
        p.qs[i] = a->q_stride[i];
        p.ks[i] = a->k_stride[i];
        p.vs[i] = a->v_stride[i];
        p.os[i] = a->o_stride[i];
    }
    return p;
}
}  // namespace

size_t fa_attention_workspace_size(const fa_params *a)
{
    if (!a) return 0;
    fa::Problem p = problem_of(a);
    // sizes, strides and dtypes only: distinct, aligned placeholder addresses
    // stand in for the pointers (never dereferenced)
    const uintptr_t base = 1024, gap = (uintptr_t)1 << 44;
    p.q = reinterpret_cast<const void *>(base);
    p.k = reinterpret_cast<const void *>(base + gap);
    p.v = reinterpret_cast<const void *>(base + 2 * gap);
    p.o = reinterpret_cast<void *>(base + 3 * gap);
    p.lse = nullptr;
    if (validate_general(p) != FA_OK) {
        clear_error();
        return 0;
    }
    if (fa::tc_supported(p)) return fa::tc_split_plan(p).workspace_bytes;
    const fa::WidePlan w = fa::wide_plan(p, 1 << 20);
    return w.ok ? w.workspace_bytes : 0;
}

fa_status fa_attention(const fa_params *a, void *workspace, size_t workspace_bytes, void *stream)
{
    clear_error();
    if (!a) return fail(FA_ERR_INVALID_ARG, "params must be non-NULL");
    const fa::Problem p = problem_of(a);
    fa_status st = validate_general(p);
    if (st != FA_OK) return st;
    return dispatch(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), 0u);
}

size_t fa_backward_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    fa::BackwardProblem p{};
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = d;
    return fa::backward_workspace_bytes(p);
}

namespace {
// A backward problem with aligned placeholder pointers and scale 1, for the
// size and plan queries (which read no pointer).
fa::BackwardProblem planning_problem(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int causal)
{
    const void *a = reinterpret_cast<const void *>(uintptr_t(256));
    void *b = reinterpret_cast<void *>(uintptr_t(256));
    return fa::BackwardProblem{a, a, a, a, a, static_cast<const float *>(a), b, b, b, B, H, N, d, 1.0f,
                               causal != 0, in_dtype, in_dtype};
}
}  // namespace

size_t fa_backward_workspace_size_ex(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype)
{
    if (B < 1 || H < 1 || N < 1 || d < 1 || (in_dtype != FA_BF16 && in_dtype != FA_FP32)) return 0;
    const fa::BackwardProblem p = planning_problem(B, H, N, d, in_dtype, 0);
    size_t n = fa::backward_workspace_bytes(p);
    if (!fa::backward_tc_supported(p) && fa::backward_wide_supported(p)) n += fa::backward_wide_copy_bytes(p);
    return n;
}

int fa_backward_plan(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int causal, size_t workspace_bytes,
                     char *desc, size_t desc_len)
{
    if (B < 1 || H < 1 || N < 1 || d < 1 || d > 1024 || (in_dtype != FA_BF16 && in_dtype != FA_FP32)) return -1;
    const fa::BackwardProblem p = planning_problem(B, H, N, d, in_dtype, causal);
    const size_t base = fa::backward_workspace_bytes(p);
    int launches;
    const char *what;
    if (fa::backward_tc_supported(p)) {
        launches = 3;
        what = "tensor-core";
    } else if (fa::backward_wide_supported(p) && workspace_bytes >= base + fa::backward_wide_copy_bytes(p)) {
        launches = in_dtype == FA_FP32 ? 4 : 3;
        what = in_dtype == FA_FP32 ? "wide-head tensor-core fp32 as bf16 hi+lo" : "wide-head tensor-core bf16";
    } else {
        launches = 3;
        what = "general";
    }
    if (desc && desc_len) snprintf(desc, desc_len, "%s", what);
    return launches;
}

fa_status fa_backward(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                      void *dq, void *dk, void *dv, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                      int causal, int in_dtype, int grad_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    clear_error();
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o, dout, lse, dq, dk, dv must be non-NULL");
    fa::Problem fwd{q, k, v, const_cast<void *>(o), nullptr, B, H, N, d, scale, causal != 0, in_dtype, in_dtype};
    if (!size_ok(fwd)) return fail(FA_ERR_INVALID_ARG, "invalid sizes or dtypes");
    if (grad_dtype != FA_BF16 && grad_dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "grad_dtype %d is not an fa_dtype", grad_dtype);
    if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    const size_t ei = dtype_size(in_dtype), eg = dtype_size(grad_dtype), n = (size_t)(B * H * N * d);
    const void *ins[5] = {q, k, v, o, dout};
    void *outs[3] = {dq, dk, dv};
    for (const void *x : ins)
        if (!aligned(x, ei)) return fail(FA_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    for (const void *x : outs)
        if (!aligned(x, eg)) return fail(FA_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    auto overlap = [](const void *a, size_t na, const void *b, size_t nb) {
        uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + nb && y < x + na;
    };
    for (int a = 0; a < 3; ++a) {
        for (const void *x : ins)
            if (overlap(outs[a], n * eg, x, n * ei)) return fail(FA_ERR_INVALID_ARG, "gradients must not overlap the inputs");
        if (overlap(outs[a], n * eg, lse, (size_t)(B * H * N) * 4))
            return fail(FA_ERR_INVALID_ARG, "gradients must not overlap the inputs");
        for (int c = a + 1; c < 3; ++c)
            if (overlap(outs[a], n * eg, outs[c], n * eg)) return fail(FA_ERR_INVALID_ARG, "dq, dk, dv must not overlap");
    }
    fa::BackwardProblem p{q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal != 0, in_dtype, grad_dtype};
    const size_t need = fa::backward_workspace_bytes(p);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned and hold %zu bytes", need);
    if (fa::backward_tc_supported(p)) {
        const char *detail = nullptr;
        cudaError_t e = fa::launch_backward_tc(p, workspace, static_cast<cudaStream_t>(stream), &detail);
        if (e != cudaSuccess)
            return detail ? fail(FA_ERR_CUDA, "tensor-core backward: %s", detail) : cuda_fail(e, "tensor-core backward");
        return FA_OK;
    }
    if (fa::backward_wide_supported(p) && workspace_bytes >= need + fa::backward_wide_copy_bytes(p)) {
        const char *detail = nullptr;
        cudaError_t e = fa::launch_backward_wide(p, workspace, static_cast<cudaStream_t>(stream), &detail);
        if (e != cudaSuccess)
            return detail ? fail(FA_ERR_CUDA, "wide-head tensor-core backward: %s", detail)
                          : cuda_fail(e, "wide-head tensor-core backward");
        return FA_OK;
    }
    cudaError_t e = fa::launch_backward_general(p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return FA_OK;
}

namespace {

// fa_forward_ws with the tensor-core kernel's query rows per work item fixed
// (0: chosen from the problem's fill)
fa_status forward_ws_rows(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t H,
                          int64_t N, int64_t d, float scale, int causal, int in_dtype, int o_dtype, void *workspace,
                          size_t workspace_bytes, void *stream, int item_rows)
{
    fa::Problem p{q, k, v, o, lse, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
    p.item_rows = item_rows;
    fa_status st = validate(p);
    if (st != FA_OK) return st;
    return dispatch(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), 0u);
}

}  // namespace

fa_status fa_forward_ws(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t H,
                        int64_t N, int64_t d, float scale, int causal, int in_dtype, int o_dtype, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    clear_error();
    return forward_ws_rows(q, k, v, o, lse, B, H, N, d, scale, causal, in_dtype, o_dtype, workspace, workspace_bytes,
                           stream, 0);
}

fa_status fa_forward_ex(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                        int64_t H, int64_t N, int64_t d, float scale, int causal, int in_dtype,
                        int o_dtype, void *stream, uint32_t flags)
{
    clear_error();
    fa::Problem p{q, k, v, o, lse, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
    fa_status st = validate(p);
    if (st != FA_OK) return st;
    return dispatch(p, nullptr, 0, static_cast<cudaStream_t>(stream), flags);
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
    return size_ok(p) ? host_layout(p).total + align256(chunk_workspace(p)) : 0;
}

fa_status fa_forward_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                          int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                          int in_dtype, int o_dtype, void *workspace, size_t workspace_bytes,
                          void *stream)
{
    clear_error();
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
    std::unique_lock<std::mutex> hold;  // the pipeline is this call's until it returns
    cudaError_t e = pipeline_res(&res, &hold);
    if (e != cudaSuccess) return cuda_fail(e, "creating the copy pipeline");
    cudaStream_t s_in = static_cast<cudaStream_t>(stream);

    const int64_t BH = B * H;
    const size_t ei = dtype_size(in_dtype), eo = dtype_size(o_dtype);
    const size_t head_elems = (size_t)(N * d);
    const int chunks = host_chunks(full);
    // every chunk runs the work items the whole problem would, so the result is
    // the device-buffer call's, bit for bit
    const int item_rows = fa::tc_item_rows(full);
    uint8_t *kernel_ws = ws + L.total;             // scratch of the wide-head path, shared by the chunks
    const size_t kernel_ws_bytes = workspace_bytes - L.total;  // (they run in order on one stream)

    // the internal streams start after earlier work on the caller's stream
    if ((e = cudaEventRecord(res->start, s_in)) != cudaSuccess) return cuda_fail(e, "event record");
    if ((e = cudaStreamWaitEvent(res->compute, res->start, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
    if ((e = cudaStreamWaitEvent(res->d2h, res->start, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");

    for (int c = 0; c < chunks; ++c) {
        const int64_t h0 = chunk_head(BH, chunks, c), h1 = chunk_head(BH, chunks, c + 1), nh = h1 - h0;
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
        fa_status st = forward_ws_rows(ws + L.q + off_in, ws + L.k + off_in, ws + L.v + off_in, ws + L.o + off_o,
                                       lse_h ? reinterpret_cast<float *>(ws + L.lse + off_l) : nullptr, 1, nh, N, d,
                                       scale, causal, in_dtype, o_dtype, kernel_ws_bytes ? kernel_ws : nullptr,
                                       kernel_ws_bytes, res->compute, item_rows);
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
    clear_error();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = take_error_words(&word, s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize / reading the device error words");
    if (word & (128u | 256u))  // the layout checks of the backward dK/dV and wide cluster kernels
        return fail(FA_ERR_CUDA, "a kernel's shared memory allocation is not aligned as its layout needs (error word 0x%x)", word);
    if (word) return fail(FA_ERR_TIMEOUT, "a device pipeline wait gave up (error word 0x%x)", word);
    return FA_OK;
}

fa_status fa_last_error(char *buf, size_t len)
{
    if (buf && len) {
        const size_t n = std::min(len - 1, g_last_error.size());
        g_last_error.copy(buf, n);
        buf[n] = '\0';
    }
    return g_last_status;
}

const char *fa_version(void) { return "0.1.0 sm_103a"; }

}  // extern "C"

namespace fa {
// Lets other translation units of the library report through fa_last_error.
void set_last_error(fa_status status, const char *msg)
{
    g_last_error = msg ? msg : "";
    g_last_status = status;
}

fa_status validate_forward(const Problem &p) { return validate(p); }
}  // namespace fa
