// Backward pass of the attention forward, by recomputation from the stored
// per-row log-sum-exp, on the CUDA cores (fp32 arithmetic), any d <= 1024.
//
// "FlashAttention" (ai360xpert.com, "Recomputation in the backward pass")
// keeps only the per-row softmax statistics from the forward pass and
// recomputes the weights tile by tile.  With LSE_i = m_i + ln l_i the weights
// are P_ij = exp(scale * q_i . k_j - LSE_i), and the gradients of
// L = sum_i dO_i . O_i are
//
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - delta_i),   delta_i = sum_j P_ij dP_ij = dO_i . O_i
//   dQ_i  = scale * sum_j dS_ij k_j
//   dK_j  = scale * sum_i dS_ij q_i
//
// Three kernels: delta per row; dK and dV per block of 64 keys (looping over
// the query blocks that see them); dQ per block of 32 queries (looping over
// the key blocks they see).  Each recomputes the 32 x 64 tiles of S and dP it
// needs, so no result is accumulated across CTAs (no atomics; deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int BR = 32;   // query rows per tile
constexpr int BC = 64;   // keys per tile
constexpr int CH = 32;   // head-dimension chunk of the S and dP products
constexpr int DCH = 64;  // output columns per CTA
constexpr int NT = 256;
constexpr int CS = CH + 1;   // padded strides
constexpr int TS = BC + 1;
constexpr int OS = DCH + 1;

__device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(p[0]); }
__device__ __forceinline__ void st(float *p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// delta_i = dO_i . O_i, one warp per row, lse2_i = LSE_i * log2(e); row i of
// head bh goes to index bh * pitch + i (pitch >= N).
template <typename T>
__global__ void fa_bwd_delta_kernel(const T *__restrict__ o, const T *__restrict__ dout, const float *__restrict__ lse,
                                    float *__restrict__ delta, float *__restrict__ lse2, int64_t rows, int d, int N,
                                    int pitch)
{
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(ld(o + row * d + c), ld(dout + row * d + c), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        const int64_t idx = (row / N) * pitch + row % N;
        delta[idx] = acc;
        lse2[idx] = lse[row] * 1.4426950408889634f;
    }
}

// The same with 16-byte loads, for rows whose length in bytes is a multiple
// of 16: 2^tpr_log2 lanes share a row (the smallest power of two that covers
// its 16-byte chunks, at most 32), so a warp reads several short rows at once.
__device__ __forceinline__ float dot16(uint4 a, uint4 b, const float *)
{
    return __uint_as_float(a.x) * __uint_as_float(b.x) + __uint_as_float(a.y) * __uint_as_float(b.y) +
           __uint_as_float(a.z) * __uint_as_float(b.z) + __uint_as_float(a.w) * __uint_as_float(b.w);
}
__device__ __forceinline__ float dot16(uint4 a, uint4 b, const __nv_bfloat16 *)
{
    const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(x[i] << 16), __uint_as_float(y[i] << 16), acc);
        acc = fmaf(__uint_as_float(x[i] & 0xffff0000u), __uint_as_float(y[i] & 0xffff0000u), acc);
    }
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(256)
fa_bwd_delta_vec_kernel(const T *__restrict__ o, const T *__restrict__ dout, const float *__restrict__ lse,
                        float *__restrict__ delta, float *__restrict__ lse2, int64_t rows, int d, int N, int pitch,
                        int tpr_log2)
{
    const int tpr = 1 << tpr_log2, chunks = d * (int)sizeof(T) / 16;
    const int sub = (int)(threadIdx.x & (uint32_t)(tpr - 1));
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> tpr_log2;
    float acc = 0.f;
    if (row < rows) {
        const uint4 *po = reinterpret_cast<const uint4 *>(o + row * d), *pg = reinterpret_cast<const uint4 *>(dout + row * d);
        for (int c = sub; c < chunks; c += tpr) acc += dot16(__ldg(po + c), __ldg(pg + c), o);
    }
    for (int off = tpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) {
        const int64_t idx = (row / N) * pitch + row % N;
        delta[idx] = acc;
        lse2[idx] = lse[row] * 1.4426950408889634f;
    }
}

// KV = true: dK, dV for one block of BC keys and one DCH-column slice.
// KV = false: dQ for one block of BR queries and one DCH-column slice.
template <typename Tin, typename Tout, bool KV>
__global__ void __launch_bounds__(NT)
fa_bwd_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
              const Tin *__restrict__ dout, const float *__restrict__ lse2, const float *__restrict__ delta,
              Tout *__restrict__ dq, Tout *__restrict__ dk, Tout *__restrict__ dv, int N, int d, int BH,
              int n_blocks, float sl, float scale, int causal)
{
    extern __shared__ float sm[];
    float *Qc = sm;                 // [BR][CS]  chunks for S and dP
    float *Kc = Qc + BR * CS;       // [BC][CS]
    float *Gc = Kc + BC * CS;       // [BR][CS]  dO chunk
    float *Vc = Gc + BR * CS;       // [BC][CS]
    float *Ps = Vc + BC * CS;       // [BR][TS]  weights
    float *Ds = Ps + BR * TS;       // [BR][TS]  dS
    float *A = Ds + BR * TS;        // KV: dO slice [BR][OS]; Q: K slice [BC][OS]
    float *Bq = A + BC * OS;        // KV: Q slice [BR][OS]

    const int tid = threadIdx.x;
    const int blk = (int)(blockIdx.x % n_blocks);
    const int bh = (int)(blockIdx.x / n_blocks);
    const int c0 = blockIdx.y * DCH;
    const int cn = min(DCH, d - c0);
    const size_t head = (size_t)bh * N * d;
    const Tin *qh = q + head, *kh = k + head, *vh = v + head, *gh = dout + head;
    const float *lh = lse2 + (size_t)bh * N, *dh = delta + (size_t)bh * N;

    const int r = tid >> 3, cg = tid & 7;  // score tile: row r, keys cg + 8u
    float acc1[16], acc2[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) acc1[x] = acc2[x] = 0.f;

    // the other side's blocks this CTA visits
    int first = 0, last;
    if (KV) {
        const int k0 = blk * BC;
        last = (N + BR - 1) / BR;
        if (causal) first = k0 / BR;  // query rows before k0 see none of these keys
    } else {
        const int q0 = blk * BR;
        last = causal ? min((N + BC - 1) / BC, (q0 + BR - 1) / BC + 1) : (N + BC - 1) / BC;
    }
    for (int it = first; it < last; ++it) {
        const int q0 = KV ? it * BR : blk * BR;
        const int k0 = KV ? blk * BC : it * BC;
        // ---- S and dP tiles (BR x BC), this thread's 8 entries
        float s[8], dp[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) s[u] = dp[u] = 0.f;
        for (int dc = 0; dc < d; dc += CH) {
            for (int e = tid; e < BR * CH; e += NT) {
                const int rr = e / CH, cc = e % CH, gr = q0 + rr, gc = dc + cc;
                const bool in = gr < N && gc < d;
                Qc[rr * CS + cc] = in ? ld(qh + (size_t)gr * d + gc) : 0.f;
                Gc[rr * CS + cc] = in ? ld(gh + (size_t)gr * d + gc) : 0.f;
            }
            for (int e = tid; e < BC * CH; e += NT) {
                const int rr = e / CH, cc = e % CH, gr = k0 + rr, gc = dc + cc;
                const bool in = gr < N && gc < d;
                Kc[rr * CS + cc] = in ? ld(kh + (size_t)gr * d + gc) : 0.f;
                Vc[rr * CS + cc] = in ? ld(vh + (size_t)gr * d + gc) : 0.f;
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < CH; ++kk) {
                const float qv = Qc[r * CS + kk], gv = Gc[r * CS + kk];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    s[u] = fmaf(qv, Kc[(cg + 8 * u) * CS + kk], s[u]);
                    dp[u] = fmaf(gv, Vc[(cg + 8 * u) * CS + kk], dp[u]);
                }
            }
            __syncthreads();
        }
        // ---- P = exp(scale s - LSE), dS = P (dP - delta)
        const int i = q0 + r;
        const float l2 = i < N ? lh[i] : 0.f, de = i < N ? dh[i] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = k0 + cg + 8 * u;
            const bool keep = i < N && j < N && (!causal || j <= i);
            const float p = keep ? exp2f(fmaf(s[u], sl, -l2)) : 0.f;
            Ps[r * TS + cg + 8 * u] = p;
            Ds[r * TS + cg + 8 * u] = p * (dp[u] - de);
        }
        // ---- output slices
        if (KV) {
            for (int e = tid; e < BR * DCH; e += NT) {
                const int rr = e / DCH, cc = e % DCH, gr = q0 + rr;
                const bool in = gr < N && cc < cn;
                A[rr * OS + cc] = in ? ld(gh + (size_t)gr * d + c0 + cc) : 0.f;
                Bq[rr * OS + cc] = in ? ld(qh + (size_t)gr * d + c0 + cc) : 0.f;
            }
        } else {
            for (int e = tid; e < BC * DCH; e += NT) {
                const int rr = e / DCH, cc = e % DCH, gr = k0 + rr;
                A[rr * OS + cc] = (gr < N && cc < cn) ? ld(kh + (size_t)gr * d + c0 + cc) : 0.f;
            }
        }
        __syncthreads();
        if (KV) {
            // key row kr = tid / 4, columns (tid % 4) + 4x
            const int kr = tid >> 2, cq = tid & 3;
#pragma unroll 4
            for (int ii = 0; ii < BR; ++ii) {
                const float p = Ps[ii * TS + kr], ds = Ds[ii * TS + kr];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    acc1[x] = fmaf(p, A[ii * OS + cq + 4 * x], acc1[x]);    // dV
                    acc2[x] = fmaf(ds, Bq[ii * OS + cq + 4 * x], acc2[x]);  // dK / scale
                }
            }
        } else {
            // query row r, columns cg + 8x
#pragma unroll 4
            for (int jj = 0; jj < BC; ++jj) {
                const float ds = Ds[r * TS + jj];
#pragma unroll
                for (int x = 0; x < 8; ++x) acc1[x] = fmaf(ds, A[jj * OS + cg + 8 * x], acc1[x]);
            }
        }
        __syncthreads();
    }
    if (KV) {
        const int kr = tid >> 2, cq = tid & 3, j = blk * BC + kr;
        if (j < N) {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int c = cq + 4 * x;
                if (c < cn) {
                    st(dv + head + (size_t)j * d + c0 + c, acc1[x]);
                    st(dk + head + (size_t)j * d + c0 + c, acc2[x] * scale);
                }
            }
        }
    } else {
        const int i = blk * BR + r;
        if (i < N) {
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int c = cg + 8 * x;
                if (c < cn) st(dq + head + (size_t)i * d + c0 + c, acc1[x] * scale);
            }
        }
    }
}

constexpr size_t SMEM_BYTES = sizeof(float) * (2 * BR * CS + 2 * BC * CS + 2 * BR * TS + BC * OS + BR * OS);

template <typename Tin, typename Tout>
cudaError_t launch_typed(const BackwardProblem &p, float *delta, float *lse2, cudaStream_t stream)
{
    const int N = (int)p.N, d = (int)p.d, BH = (int)(p.B * p.H);
    const int64_t rows = (int64_t)BH * N;
    fa_bwd_delta_kernel<Tin><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const Tin *>(p.o), static_cast<const Tin *>(p.dout), p.lse, delta, lse2, rows, d, N, N);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const float sl = p.scale * 1.4426950408889634f;
    const unsigned nslices = (unsigned)((d + DCH - 1) / DCH);
    auto kv = fa_bwd_kernel<Tin, Tout, true>;
    auto qk = fa_bwd_kernel<Tin, Tout, false>;
    if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(qk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)) != cudaSuccess)
        return e;
    const int nkb = (N + BC - 1) / BC, nqb = (N + BR - 1) / BR;
    const Tin *q = static_cast<const Tin *>(p.q), *k = static_cast<const Tin *>(p.k), *v = static_cast<const Tin *>(p.v),
              *g = static_cast<const Tin *>(p.dout);
    Tout *dq = static_cast<Tout *>(p.dq), *dk = static_cast<Tout *>(p.dk), *dv = static_cast<Tout *>(p.dv);
    kv<<<dim3((unsigned)((int64_t)nkb * BH), nslices), NT, SMEM_BYTES, stream>>>(q, k, v, g, lse2, delta, dq, dk, dv, N,
                                                                               d, BH, nkb, sl, p.scale, p.causal);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    qk<<<dim3((unsigned)((int64_t)nqb * BH), nslices), NT, SMEM_BYTES, stream>>>(q, k, v, g, lse2, delta, dq, dk, dv, N,
                                                                               d, BH, nqb, sl, p.scale, p.causal);
    return cudaGetLastError();
}

}  // namespace

// delta and lse2 arrays, each [B*H][N rounded up to 128] floats (the tensor-
// core backward reads them in 128-row blocks).
size_t backward_workspace_bytes(const BackwardProblem &p)
{
    const size_t rows = (size_t)(p.B * p.H) * (size_t)((p.N + 127) / 128 * 128);
    return 2 * ((rows * 4 + 255) & ~size_t(255));
}

cudaError_t launch_backward_delta(const BackwardProblem &p, void *workspace, cudaStream_t stream, int pitch,
                                  float **delta_out, float **lse2_out)
{
    const size_t rows_pad = (size_t)(p.B * p.H) * (size_t)((p.N + 127) / 128 * 128);
    float *delta = static_cast<float *>(workspace);
    float *lse2 = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ((rows_pad * 4 + 255) & ~size_t(255)));
    *delta_out = delta;
    *lse2_out = lse2;
    const int64_t rows = p.B * p.H * p.N;
    const int64_t row_bytes = p.d * (p.in_dtype == 0 ? 2 : 4);
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    if (row_bytes % 16 == 0 && al16(p.o) && al16(p.dout)) {
        int tpr_log2 = 0;
        while ((1 << tpr_log2) < 32 && (int64_t)(1 << tpr_log2) * 16 < row_bytes) ++tpr_log2;
        const unsigned blocks = (unsigned)((rows * (1 << tpr_log2) + 255) / 256);
        if (p.in_dtype == 0)
            fa_bwd_delta_vec_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(p.o), static_cast<const __nv_bfloat16 *>(p.dout), p.lse, delta, lse2,
                rows, (int)p.d, (int)p.N, pitch, tpr_log2);
        else
            fa_bwd_delta_vec_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(p.o),
                                                                        static_cast<const float *>(p.dout), p.lse, delta,
                                                                        lse2, rows, (int)p.d, (int)p.N, pitch, tpr_log2);
        return cudaGetLastError();
    }
    if (p.in_dtype == 0)
        fa_bwd_delta_kernel<__nv_bfloat16><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(p.o), static_cast<const __nv_bfloat16 *>(p.dout), p.lse, delta, lse2,
            rows, (int)p.d, (int)p.N, pitch);
    else
        fa_bwd_delta_kernel<float><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
            static_cast<const float *>(p.o), static_cast<const float *>(p.dout), p.lse, delta, lse2, rows, (int)p.d,
            (int)p.N, pitch);
    return cudaGetLastError();
}

cudaError_t launch_backward_general(const BackwardProblem &p, void *workspace, cudaStream_t stream)
{
    const size_t rows_pad = (size_t)(p.B * p.H) * (size_t)((p.N + 127) / 128 * 128);
    float *delta = static_cast<float *>(workspace);
    float *lse2 = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ((rows_pad * 4 + 255) & ~size_t(255)));
    const bool in_bf16 = p.in_dtype == 0, g_bf16 = p.grad_dtype == 0;
    if (in_bf16 && g_bf16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(p, delta, lse2, stream);
    if (in_bf16) return launch_typed<__nv_bfloat16, float>(p, delta, lse2, stream);
    if (g_bf16) return launch_typed<float, __nv_bfloat16>(p, delta, lse2, stream);
    return launch_typed<float, float>(p, delta, lse2, stream);
}

}  // namespace fa
