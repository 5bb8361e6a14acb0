// Internal interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// One forward problem, already validated by the C ABI.
//   Q [B, H, N, d], K [B, H, Nk, d], V [B, H, Nk, dv], O [B, H, N, dv],
//   LSE [B, H, N] contiguous.  Nk = 0 means N, dv = 0 means d.  Strides are
//   in elements for (batch, head, sequence), the head dimension contiguous;
//   all-zero strides mean the contiguous layout.
struct Problem {
    const void *q, *k, *v;
    void *o;
    float *lse;            // may be null
    int64_t B, H, N, d;
    float scale;
    int causal;
    int in_dtype;          // fa_dtype
    int o_dtype;           // fa_dtype
    int64_t Nk = 0, dv = 0;
    int64_t qs[3] = {0, 0, 0}, ks[3] = {0, 0, 0}, vs[3] = {0, 0, 0}, os[3] = {0, 0, 0};
    // tensor-core kernel: query rows per work item, 128 or 256; 0 = chosen from
    // the problem's own fill (tc_item_rows).  A caller that runs a problem in
    // pieces fixes it so that every piece computes as the whole would.
    int item_rows = 0;
};

inline int64_t keys_of(const Problem &p) { return p.Nk ? p.Nk : p.N; }
inline int64_t dv_of(const Problem &p) { return p.dv ? p.dv : p.d; }

// Element strides (batch, head, sequence) of tensor t: 0 = Q, 1 = K, 2 = V, 3 = O.
inline void strides_of(const Problem &p, int t, int64_t out[3])
{
    const int64_t *s = t == 0 ? p.qs : t == 1 ? p.ks : t == 2 ? p.vs : p.os;
    if (s[0] || s[1] || s[2]) {
        out[0] = s[0];
        out[1] = s[1];
        out[2] = s[2];
        return;
    }
    const int64_t n = (t == 0 || t == 3) ? p.N : keys_of(p);
    const int64_t w = (t <= 1) ? p.d : dv_of(p);
    out[0] = p.H * n * w;
    out[1] = n * w;
    out[2] = w;
}

// True when every tensor has the contiguous layout and Nk = N, dv = d.
inline bool plain_layout(const Problem &p)
{
    for (int t = 0; t < 4; ++t) {
        const int64_t *s = t == 0 ? p.qs : t == 1 ? p.ks : t == 2 ? p.vs : p.os;
        if (s[0] || s[1] || s[2]) {
            int64_t c[3];
            Problem z = p;
            z.qs[0] = z.qs[1] = z.qs[2] = 0;
            z.ks[0] = z.ks[1] = z.ks[2] = 0;
            z.vs[0] = z.vs[1] = z.vs[2] = 0;
            z.os[0] = z.os[1] = z.os[2] = 0;
            strides_of(z, t, c);
            if (s[0] != c[0] || s[1] != c[1] || s[2] != c[2]) return false;
        }
    }
    return keys_of(p) == p.N && dv_of(p) == p.d;
}

// General-d CUDA-core kernel (any d <= 1024, bf16 or fp32 in and out).
cudaError_t launch_general(const Problem &p, cudaStream_t stream);

// Tensor-core kernel (tcgen05 + TMA): bf16 in, d in {64, 128}.
bool tc_supported(const Problem &p);
// Returns cudaSuccess or an error; *detail receives a static description on
// failures that are not CUDA errors (tensor-map encoding).
cudaError_t launch_tc(const Problem &p, cudaStream_t stream, uint32_t flags, const char **detail);

// Device address of the error word of the tensor-core kernel (ORed bits of
// waits that gave up; cleared by the host after reading).
cudaError_t tc_error_word_ptr(uint32_t **ptr);

// Wide-head tensor-core path (fa_wide.cu): fp32 inputs with d % 128 == 0
// (d <= 1024), bf16 inputs with d % 128 == 0 and 256 <= d <= 1024.
struct WidePlan {
    bool ok;             // the path applies to this problem
    int nprod;           // 3: fp32 inputs as bf16 hi + lo pairs; 1: bf16 inputs
    int dv;              // width of the O slice a CTA owns (256 or 128)
    int cluster;         // CTAs per cluster sharing one formation of S (d / 256 for d = 512, 1024), else 1
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
cudaError_t wide_error_word_ptr(uint32_t **ptr);
// Merge of key-range partials (fa_wide.cu): per split s, unnormalised O rows
// o_part[s][row][D] (fp32), the row's reference maximum m_part (log2 units),
// its exact weight sum l_part and its bf16-rounding correction d_part, rows =
// BH * N; writes O (contiguous [BH * N][D]) and LSE.  n_split <= 16.
cudaError_t launch_combine(const float *o_part, const float *m_part, const float *l_part, const float *d_part, void *o,
                           bool o_fp32, float *lse, int64_t BH, int64_t N, int D, int n_split, cudaStream_t stream);

// Key-range split of the tensor-core kernel (fa_tc.cu) for problems with too
// few work items to fill the GPU: unmasked, O contiguous; n_split <= 1 means
// no split.  The partials need `workspace_bytes`.
struct TcSplit {
    int n_split, kv_per;
    size_t workspace_bytes;
};
TcSplit tc_split_plan(const Problem &p);
// Query rows per work item of the tensor-core kernel: 256 (two query tiles),
// or 128 (one tile, its key tiles shared by both softmax warpgroups) for
// unmasked problems of at most 128 query rows or too few items to fill the GPU.
int tc_item_rows(const Problem &p);
cudaError_t launch_tc_split(const Problem &p, const TcSplit &sp, void *workspace, cudaStream_t stream, const char **detail);

// Backward problem: contiguous [B, H, N, d] Q, K, V, O, dO of in_dtype,
// LSE [B, H, N] fp32 from the forward pass, gradients of grad_dtype.
struct BackwardProblem {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int64_t B, H, N, d;
    float scale;
    int causal;
    int in_dtype, grad_dtype;
};
size_t backward_workspace_bytes(const BackwardProblem &p);
cudaError_t launch_backward_general(const BackwardProblem &p, void *workspace, cudaStream_t stream);
// delta and lse2 (LSE * log2 e) into the workspace with the given row pitch per head.
cudaError_t launch_backward_delta(const BackwardProblem &p, void *workspace, cudaStream_t stream, int pitch,
                                  float **delta, float **lse2);
// Tensor-core backward: bf16 inputs, d in {64, 128}, scale > 0, 16-byte aligned.
bool backward_tc_supported(const BackwardProblem &p);
cudaError_t launch_backward_tc(const BackwardProblem &p, void *workspace, cudaStream_t stream, const char **detail);
cudaError_t bwd_error_word_ptr(uint32_t **ptr);
// Wide-head tensor-core backward (fa_backward_wide.cu): d % 128 == 0, d <= 1024,
// bf16 inputs with d >= 256, fp32 inputs (as bf16 hi + lo) with d >= 128.
// fp32 inputs need backward_wide_copy_bytes more workspace after the
// backward_workspace_bytes of the row vectors.
bool backward_wide_supported(const BackwardProblem &p);
size_t backward_wide_copy_bytes(const BackwardProblem &p);
cudaError_t launch_backward_wide(const BackwardProblem &p, void *workspace, cudaStream_t stream, const char **detail);
cudaError_t bwdw_error_word_ptr(uint32_t **ptr);
// x = hi + lo with hi = bf16(x), lo = bf16(x - hi) for `count` (<= 4) fp32
// arrays of n elements each (n % 4 == 0, 16-byte aligned), one launch.
cudaError_t launch_split_hilo(const float *const *x, void *const *hi, void *const *lo, int count, size_t n,
                              cudaStream_t stream);

// Sets the status and text fa_last_error returns on this host thread.
void set_last_error(fa_status status, const char *msg);

// The argument rules of fa_forward / fa_forward_ws (pointers, alignment,
// sizes, dtypes, scale, overlaps); FA_OK or the failure, reported through
// fa_last_error.
fa_status validate_forward(const Problem &p);

}  // namespace fa
