/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward pass.
 *
 * The operation is the one every page on the subject defines:
 *
 *     O = softmax(Q K^T * scale) V,   softmax taken row by row over the keys,
 *
 * ("Deep Learning - Flash Attention", "Refresher - Softmax of a Matrix
 * Normalizes Each Row"; "The Details of Flash Attention", "The Attention
 * Computation"), computed tile by tile with the online-softmax recurrence
 * (running row maximum m, running denominator l, rescale factor
 * alpha = exp(m_old - m_new)) of "The Details of Flash Attention", "Online
 * Softmax" and "Tiling the Loop", so that the N x N score matrix never
 * reaches global memory.  The result is exact up to floating-point rounding
 * ("FlashAttention", ai360xpert.com, "Show Me the Code").
 *
 * Conventions shared by every entry point:
 *   - Q, K, V and O are contiguous row-major [B, H, N, d] tensors (batch,
 *     head, sequence, head dimension), the (B, nhead, N, nd) shape of "The
 *     Details of Flash Attention", "The Attention Computation".  Batch and
 *     head are independent problems.
 *   - LSE is a contiguous [B, H, N] float32 tensor:
 *     LSE[b,h,i] = ln sum_j exp(scale * q_i . k_j), i.e. m_i + ln l_i in
 *     natural-log units of the scaled scores -- the per-row softmax
 *     statistics that "FlashAttention" (ai360xpert.com, "Recomputation in
 *     the backward pass") keeps instead of the weights.
 *   - causal != 0 masks key j > query i (the mask of "PyTorch
 *     Implementation" in "Transformer Attention: A Mathematical Deep Dive");
 *     key tiles that lie wholly above the diagonal are skipped.
 *   - The caller owns every buffer, workspaces included.  The library
 *     allocates no device memory and keeps no per-call state; it caches one
 *     driver entry point and, for fa_forward_host, two streams and some
 *     events per device.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void *;
 *     NULL = the legacy default stream).  Streams travel as void * and dtypes
 *     as int (fa_dtype values) so that this header includes no CUDA header and
 *     a plain C program can use it.  Argument errors are reported before anything is
 *     launched; launch errors are reported on return; a device-side timeout
 *     (a pipeline wait that gave up) is reported by fa_check_device_error.
 *   - There is no CPU fallback: a shape or dtype no kernel covers returns
 *     FA_ERR_UNSUPPORTED.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, bad size, non-finite scale */
    FA_ERR_UNSUPPORTED = 2,   /* valid arguments that no kernel here covers */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (text in fa_last_error) */
    FA_ERR_TIMEOUT = 4        /* a device pipeline wait gave up (see fa_check_device_error) */
} fa_status;

typedef enum fa_dtype {
    FA_BF16 = 0,              /* bfloat16 storage */
    FA_FP32 = 1               /* float32 storage */
} fa_dtype;

/* fa_forward_ex flags */
#define FA_FLAG_GENERAL_PATH 0x1u  /* run the general-d CUDA-core kernel even where
                                      the tensor-core kernel applies */
/* Fault injection for tests of the failure path: the tensor-core kernel's
 * loader never issues the load of key tile 1, and every pipeline wait gives up
 * after 20 ms instead of 2 s.  The waits that depend on that tile run out, the
 * kernel frees its tensor memory and exits, and fa_check_device_error reports
 * FA_ERR_TIMEOUT; nothing traps, faults or hangs, and the next call works.
 * Has no effect when N <= 128 or when the general-d kernel runs. */
#define FA_FLAG_TEST_SKIP_KV_LOAD 0x100u

/*
 * fa_forward -- O (and LSE) of one attention forward pass.
 *
 *   q, k, v   device pointers, [B, H, N, d] elements of `in_dtype`.
 *   o         device pointer, [B, H, N, d] elements of `o_dtype`; written.
 *   lse       device pointer to [B, H, N] float32, or NULL to skip it.
 *   B, H, N   >= 1; B * H * N < 2^31.   d: 1 <= d <= 1024.
 *   scale     finite; pass 1/sqrt(d) for the usual 1/sqrt(d_k) scaling.
 *   causal    0 or non-zero (mask key j > query i).
 *   in_dtype, o_dtype   fa_dtype values.
 *   stream    cudaStream_t to enqueue on.
 *
 * Pointers must be aligned to their element size.  The tensor-core kernel is
 * used when in_dtype = FA_BF16, d is a multiple of 8 up to 128 (64 and 128
 * natively, other widths padded inside the kernel to 64 or 128 with zero
 * columns), scale > 0 and q, k, v, o are 16-byte aligned; bf16 inputs with d a
 * multiple of 128 in 256..1024 take the wide-head tensor-core path; everything
 * else the general-d kernel.  Outputs are undefined if the
 * call does not return FA_OK.  O must not overlap Q, K, V or LSE.
 */
fa_status fa_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                     int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                     int in_dtype, int o_dtype, void *stream);

/* fa_forward with FA_FLAG_* bits in `flags` (0 = fa_forward). */
fa_status fa_forward_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                        int in_dtype, int o_dtype, void *stream, uint32_t flags);

/*
 * fa_workspace_size -- bytes of device workspace that let fa_forward_ws run
 * this problem at full parallelism.  On the wide-head tensor-core path: the
 * bf16 hi/lo copies of fp32 inputs and, when the key range is split across
 * CTAs, the per-split partial O, m and l that a combine step merges with
 * the rule of "FlashAttention Engine: Hardware-Aware Exact Attention & SRAM
 * Tiling" ("Core FlashAttention Mechanics", item 3).  On the 64/128
 * tensor-core kernel: the same partials when the problem has too few
 * 256-row query blocks to fill the GPU (no mask, long key range), so that
 * CTAs split the keys.  0 means the problem needs none.
 */
size_t fa_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype, int causal);

/*
 * fa_plan -- the kernel path fa_forward_ws would take for this problem with
 * `workspace_bytes` of workspace (0 = none, as fa_forward): returns the
 * number of kernel launches one call enqueues (-1 for invalid sizes) and
 * writes a short description ("tensor-core d=128", "wide-head ...",
 * "general-d") into desc (may be NULL).  Pointer alignment is assumed.
 * A tensor-core description ends in ", one query tile per item" when the
 * kernel's work items are single 128-row query tiles rather than 256-row
 * blocks: unmasked problems of at most 128 query rows, and unmasked problems
 * whose 256-row blocks would occupy at most half of the device's SMs.
 */
int fa_plan(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype, int causal,
            size_t workspace_bytes, char *desc, size_t desc_len);

/*
 * fa_forward_ws -- fa_forward with a caller-owned device workspace
 * (256-byte aligned, contents unspecified on return; must not be used by
 * anything else until the call's work on `stream` has finished).
 *
 * With workspace_bytes >= fa_workspace_size(...) the wide-head path
 * (fp32 inputs with d % 128 == 0, bf16 inputs with d in {256, 384, ... 1024})
 * runs on the tensor cores, fp32 operands carried as bf16 hi + lo pairs.
 * With less (or NULL) it runs with fewer splits, or on the general-d kernel
 * when fp32 inputs leave no room for their bf16 copies.  fa_forward uses
 * the wide path only where it needs no workspace (bf16 inputs).
 */
fa_status fa_forward_ws(const void *q, const void *k, const void *v, void *o, float *lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                        int in_dtype, int o_dtype, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * fa_host_workspace_size -- bytes of device workspace fa_forward_host needs
 * for this problem (device copies of Q, K, V, O and LSE, 256-byte aligned
 * each, plus the wide-head path's scratch for one chunk of heads).  Returns 0
 * for arguments fa_forward would reject.
 */
size_t fa_host_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int o_dtype);

/*
 * fa_forward_host -- the same forward pass on HOST buffers, end to end.
 *
 *   q_h, k_h, v_h  host pointers, [B, H, N, d] elements of `in_dtype`
 *                  (page-locked memory lets the copies overlap the kernels).
 *   o_h            host pointer, [B, H, N, d] elements of `o_dtype`; written.
 *   lse_h          host pointer to [B, H, N] float32, or NULL.
 *   workspace      device pointer, >= fa_host_workspace_size(...) bytes,
 *                  256-byte aligned, owned by the caller; its contents on
 *                  return are unspecified.
 *   the rest       as fa_forward.
 *
 * The heads are split into up to 8 chunks; chunk c's host-to-device copy
 * (on `stream`), its kernel and its device-to-host copy (on two streams the
 * library creates once per device) form a pipeline, so copies in both
 * directions overlap the compute of other chunks.  The call is synchronous:
 * it returns once o_h and lse_h hold the result, or with the first error
 * (a device-side timeout included).  Concurrent calls on one device (from
 * several host threads) take turns: the pipeline streams are one call's at a
 * time.
 */
fa_status fa_forward_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                          int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                          int in_dtype, int o_dtype, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * fa_attention -- the general form: cross-attention shapes and strided
 * layouts ("Transformer Attention: A Mathematical Deep Dive", "The Attention
 * Formula": Q is (n, d_k), K is (m, d_k), V is (m, d_v) per head).
 *
 *   Q [B, H, Nq, dk], K [B, H, Nk, dk], V [B, H, Nk, dv], O [B, H, Nq, dv];
 *   element (b, h, n, c) of a tensor lives at ptr + b*s[0] + h*s[1] + n*s[2] + c
 *   (elements, the last dimension contiguous); an all-zero stride triple means
 *   the contiguous layout.  The (batch, seq, heads, dim) layout of the
 *   flash_attn_func usage is s = {N*H*d, d, H*d}.  Strides must be >= 0;
 *   O's must not make two of its elements share an address.
 *   LSE is a contiguous [B, H, Nq] float32 tensor or NULL.
 *   causal masks key j > query i (the same rule as for Nq = Nk).
 *   workspace as for fa_forward_ws (may be NULL).
 *
 * The tensor-core kernel covers bf16 inputs with dk and dv each a multiple
 * of 8 up to 128, scale > 0, 16-byte aligned pointers and every stride a
 * non-zero multiple of 16 bytes; the wide-head path covers the contiguous Nq = Nk,
 * dk = dv layouts of fa_forward_ws; the general-d kernel covers the rest
 * (dk, dv <= 1024, any strides).
 */
typedef struct fa_params {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t B, H, Nq, Nk, dk, dv;
    int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];
    float scale;
    int causal;
    int in_dtype, o_dtype;
} fa_params;

fa_status fa_attention(const fa_params *p, void *workspace, size_t workspace_bytes, void *stream);

/*
 * fa_attention_workspace_size -- bytes of device workspace that let
 * fa_attention run `p` at full parallelism (the key-range partials described
 * under fa_workspace_size; a shorter workspace runs it without the split).
 * Reads only the sizes, strides and dtypes of *p.  0 for none or for an
 * invalid *p.
 */
size_t fa_attention_workspace_size(const fa_params *p);

/*
 * fa_backward_workspace_size / fa_backward -- gradients of the forward pass
 * by recomputation from the stored per-row statistics ("FlashAttention",
 * ai360xpert.com, "Recomputation in the backward pass"): with
 * P_ij = exp(scale q_i.k_j - LSE_i) and L = sum_i dO_i . O_i,
 *   dV = P^T dO,  dS = P o (dO V^T - delta),  delta_i = dO_i . O_i,
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   q, k, v, o, dout  device pointers, contiguous [B, H, N, d] of in_dtype
 *                     (o is the forward output, dout the gradient of O).
 *   lse               device pointer, [B, H, N] fp32 from the forward pass.
 *   dq, dk, dv        device pointers, [B, H, N, d] of grad_dtype; written.
 *   workspace         device pointer, >= fa_backward_workspace_size bytes,
 *                     256-byte aligned (per-row delta and LSE in log2 units).
 *   scale, causal     as in the forward call that produced o and lse.
 * Asynchronous on `stream`; no result is accumulated across CTAs, so the
 * gradients are deterministic.  Gradients must not overlap the inputs.
 */
size_t fa_backward_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d);
fa_status fa_backward(const void *q, const void *k, const void *v, const void *o, const void *dout,
                      const float *lse, void *dq, void *dk, void *dv,
                      int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                      int in_dtype, int grad_dtype, void *workspace, size_t workspace_bytes,
                      void *stream);

/*
 * fa_backward_workspace_size_ex -- the workspace fa_backward needs to run this
 * problem on the tensor cores.  fp32 inputs with d a multiple of 128 (up to
 * 1024) take the wide-head tensor-core backward, which carries them as bf16
 * hi + lo pairs (as the wide forward does) and needs room for those copies of
 * Q, K, V and dO; with only fa_backward_workspace_size bytes they run on the
 * CUDA cores.  For every other problem it equals fa_backward_workspace_size.
 * 0 for invalid sizes or dtypes.
 *
 * The tensor-core backward covers bf16 inputs with d a multiple of 8 up to
 * 128 (64 and 128 natively; a narrower head is padded with zero columns up to
 * the next of them, and only its own columns are written), and, for
 * head dimensions too wide for one tile's gradients to fit tensor memory, bf16
 * inputs with d a multiple of 128 in 256..1024 and fp32 inputs with d a
 * multiple of 128 in 128..1024: a CTA owns a slice of the gradient columns
 * and forms the score products S and dP over the whole head dimension
 * itself.  Everything else runs on the CUDA cores.  All of them need
 * scale > 0 and 16-byte aligned pointers for the tensor cores.
 */
size_t fa_backward_workspace_size_ex(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype);

/*
 * fa_backward_plan -- the path fa_backward would take for this problem with
 * `workspace_bytes` of workspace: returns the number of kernel launches one
 * call enqueues (-1 for invalid sizes) and writes a short description
 * ("tensor-core", "wide-head tensor-core ...", "general") into desc (may be
 * NULL).  Pointer alignment and scale > 0 are assumed.
 */
int fa_backward_plan(int64_t B, int64_t H, int64_t N, int64_t d, int in_dtype, int causal, size_t workspace_bytes,
                     char *desc, size_t desc_len);

/*
 * fa_forward_noalloc -- the wide-head path of fa_forward_ws for callers that
 * cannot allocate device memory.  The pages have no counterpart: it exists
 * for code that must not call cudaMalloc while it runs (a plugin inside a
 * framework that owns all device memory through its own allocator, or a
 * service that plans its memory up front because a run-time allocation can
 * stall the device or fail under memory pressure).
 *
 * Arguments, layouts and the result are those of fa_forward; the caller
 * still owns Q, K, V, O and LSE.  The scratch comes from a device array of
 * FA_NOALLOC_SCRATCH_BYTES inside this library, which every GPU that loads
 * the library holds until the process exits.  The call allocates nothing.
 *   - Covers the wide-head path only: fp32 inputs with d a multiple of 128,
 *     or bf16 inputs with d a multiple of 128 in 256..1024 (scale > 0,
 *     16-byte aligned pointers).  Other problems return FA_ERR_UNSUPPORTED:
 *     fa_forward needs no scratch for them.
 *   - A problem whose scratch exceeds FA_NOALLOC_SCRATCH_BYTES (after falling
 *     back to a single key split) returns FA_ERR_UNSUPPORTED with the sizes
 *     in fa_last_error.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing needs to start at zero).  Calls whose work can
 *     overlap on the GPU race on it: order them, e.g. on one stream.
 *   - Arguments are checked by the rules of fa_forward_ws.
 *   - The first call on a device looks up the array's address with that
 *     device current and keeps it with the identity of the device's context;
 *     a later call that finds another context (after cudaDeviceReset, for
 *     instance) looks it up again.  Make the first call, and the first call
 *     after a reset, before any stream capture begins.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
fa_status fa_forward_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                             int in_dtype, int o_dtype, void *stream);

/*
 * fa_check_device_error -- synchronise `stream`, then read and clear the
 * device-side error word the kernels set when a bounded pipeline wait gives
 * up.  Returns FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if the stream itself
 * reports an error (or a backward kernel found its shared-memory allocation
 * unusable for its layout and did nothing).  The error words are one per kernel family on the
 * current device, not per stream: a wait that gave up in work on another
 * stream is reported (and cleared) by whichever check reads the words
 * first once that work has run.
 */
fa_status fa_check_device_error(void *stream);

/*
 * fa_last_error -- the status and text of the last fa_* call on the calling
 * host thread that can fail.
 *
 *   buf, len  caller-owned host buffer of len bytes that receives the text,
 *             NUL-terminated and cut to len - 1 characters ("" when that call
 *             succeeded); NULL or len = 0 copies nothing.
 * Returns the status that call returned (FA_OK when it succeeded).  Each
 * thread keeps its own record; every entry point but fa_last_error,
 * fa_version and the size queries replaces it.
 */
fa_status fa_last_error(char *buf, size_t len);

/* Library version string, e.g. "0.1.0 sm_103a". */
const char *fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
