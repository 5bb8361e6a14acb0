// fa_forward_noalloc: the wide-head tensor-core path with its scratch in a
// fixed device array of this library instead of a caller workspace.
//
// Who needs it: code that must not allocate device memory while it runs --
// a plugin living inside a framework that owns the GPU's memory through its
// own allocator and forbids direct cudaMalloc calls, or a latency-critical
// service that plans all its memory up front because an allocation at run
// time can stall the device, fragment the heap or fail under memory
// pressure.  Such callers still provide Q, K, V, O and LSE; the scratch the
// wide-head path needs (bf16 hi/lo copies of fp32 inputs and the per-split
// partial results) comes from `g_noalloc_scratch` below.
//
// Costs and rules:
//   * every GPU that loads this library holds FA_NOALLOC_SCRATCH_BYTES of
//     device memory for the array until the process exits;
//   * arguments are checked by the same rules as fa_forward_ws;
//   * problems whose scratch does not fit are rejected (FA_ERR_UNSUPPORTED,
//     with the sizes in fa_last_error); nothing falls back to allocating;
//   * all calls on a device share its one array, which keeps whatever the
//     last call left there.  Nothing in it has to start at zero: every value
//     the kernels read was written earlier in the same call.  Calls whose
//     work can overlap on the GPU (issued on different streams with nothing
//     ordering them) race on the array, so callers must order them, for
//     example by issuing them all on one stream.  Each device has its own
//     copy of the array;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it with the
//     identity of the device's context.  A call that finds another context
//     current (after cudaDeviceReset, for instance, the module is loaded
//     again and the array may sit elsewhere) looks the address up again.
//     Make the first call, and the first call after a reset, before any
//     stream capture begins.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
struct ScratchEntry {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void *ptr;
};
ScratchEntry g_scratch[MAX_DEVICES];
std::mutex g_scratch_mu;

fa_status report(fa_status st, const char *fmt, ...)
{
    char buf[320];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    fa::set_last_error(st, buf);
    return st;
}

// Unique id of the calling thread's current context (cuCtxGetId; ids are
// never reused within a process), or 0 when no context is current yet.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

bool current_context_id(unsigned long long *id)
{
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext c = nullptr;
    *id = 0;
    if (get_current(&c) != CUDA_SUCCESS) return false;
    if (!c) return true;
    return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of the current device's scratch array: looked up once per
// device and context, then taken from the cache.
fa_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES) return report(FA_ERR_UNSUPPORTED, "device %d is beyond the %d supported", dev, MAX_DEVICES);
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return report(FA_ERR_CUDA, "cannot read the identity of the current context");
    std::lock_guard<std::mutex> g(g_scratch_mu);
    ScratchEntry &s = g_scratch[dev];
    if (ctx == 0 || s.ptr == nullptr || s.ctx_id != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with no context yet, this creates it
        if (e != cudaSuccess || !p)
            return report(FA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
        if (!current_context_id(&ctx) || ctx == 0)
            return report(FA_ERR_CUDA, "cannot read the identity of the current context");
        s.ctx_id = ctx;
        s.ptr = p;
    }
    *out = s.ptr;
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_forward_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                        int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                                        int in_dtype, int o_dtype, void *stream)
{
    fa::set_last_error(FA_OK, "");
    fa::Problem p{q, k, v, o, lse, B, H, N, d, scale, causal != 0, in_dtype, o_dtype};
    const fa_status valid = fa::validate_forward(p);
    if (valid != FA_OK) return valid;

    fa::WidePlan w = fa::wide_plan(p, 1 << 20);
    if (!w.ok)
        return report(FA_ERR_UNSUPPORTED,
                      "fa_forward_noalloc covers the wide-head path only (fp32 inputs with d a multiple of 128, "
                      "bf16 inputs with d a multiple of 128 in 256..1024, scale > 0, 16-byte aligned pointers); "
                      "fa_forward allocates nothing for other problems");
    if (w.workspace_bytes > (size_t)FA_NOALLOC_SCRATCH_BYTES) w = fa::wide_plan(p, 1);  // no partials
    if (w.workspace_bytes > (size_t)FA_NOALLOC_SCRATCH_BYTES)
        return report(FA_ERR_UNSUPPORTED, "this problem needs %zu bytes of scratch, above the %zu-byte maximum",
                      w.workspace_bytes, (size_t)FA_NOALLOC_SCRATCH_BYTES);

    void *scratch = nullptr;
    fa_status st = scratch_address(&scratch);
    if (st != FA_OK) return st;
    const char *detail = nullptr;
    cudaError_t e = fa::launch_wide(p, w, w.workspace_bytes ? scratch : nullptr, static_cast<cudaStream_t>(stream),
                                    0u, &detail);
    if (e != cudaSuccess)
        return detail ? report(FA_ERR_CUDA, "wide-head launch: %s", detail)
                      : report(FA_ERR_CUDA, "wide-head launch: %s", cudaGetErrorString(e));
    return FA_OK;
}
