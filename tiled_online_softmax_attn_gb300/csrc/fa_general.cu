// General-d attention forward on the CUDA cores (fp32 arithmetic).
//
// Covers every head dimension up to 1024 and both storage types, including
// the single-head d = 1024 fp32 shape of the CUDA walkthrough in "The
// Details of Flash Attention".  It is the same tiled online-softmax
// recurrence as the tensor-core kernel ("The Details of Flash Attention",
// "Tiling the Loop"; "Deep Learning - Flash Attention", "An Example",
// steps 4-6), in the unnormalised form: O and l are rescaled by
// alpha = 2^(m_old - m_new) whenever a key tile raises the running maximum,
// and O is divided by l once after the last tile.
//
// Work decomposition (one CTA of 256 threads):
//   * a block of BR = 32 query rows of one (batch, head) and one chunk of
//     DV = 128 output columns -- query blocks are independent ("An
//     Example", step 7); a head dimension above 128 is split across CTAs,
//     each recomputing the scores for its rows;
//   * key/value tiles of BC = 64 keys streamed through shared memory, the
//     score tile Q_i K_j^T accumulated over the head dimension in chunks of
//     DK = 32 columns;
//   * 8 threads per query row: each holds 8 scores of the tile and 16
//     output columns; the row max and row sum use 3 xor-shuffles inside
//     the 8-lane group.
// Scores are kept in log2 units (scale * log2 e folded in), so each weight
// is one exp2 of (s - m).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int BR = 32;    // query rows per CTA
constexpr int BC = 64;    // keys per tile
constexpr int DK = 32;    // head-dimension chunk of the score product
constexpr int DV = 128;   // output columns per CTA
constexpr int NT = 256;   // threads per CTA
constexpr int QS = DK + 1;  // padded strides (no bank conflicts)
constexpr int PS = BC + 1;
constexpr size_t SMEM_BYTES = sizeof(float) * (BR * QS + BC * QS + BR * PS + BC * DV + BR);

__device__ __forceinline__ float load_f(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load_f(const __nv_bfloat16 *p) { return __bfloat162float(p[0]); }
__device__ __forceinline__ void store_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float group8_max(float x) {
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}
__device__ __forceinline__ float group8_sum(float x) {
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Element strides (batch, head, row) of the four tensors; the last dimension
// is contiguous.
struct Strides {
    int64_t q[3], k[3], v[3], o[3];
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NT)
fa_general_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                  Tout *__restrict__ o, float *__restrict__ lse, int N, int Nk, int d, int dv, int H,
                  int n_qblocks, int BH, float scale_log2, int causal, const Strides st)
{
    extern __shared__ float smem[];
    float *Qs = smem;              // [BR][QS]  query chunk
    float *Ks = Qs + BR * QS;      // [BC][QS]  key chunk
    float *Ps = Ks + BC * QS;      // [BR][PS]  weights of the current tile
    float *Vs = Ps + BR * PS;      // [BC][DV]  value tile, this CTA's columns

    const int tid = threadIdx.x;
    int qb, bh;
    if (causal) {  // longest rows first: the last query blocks see the most keys
        qb = n_qblocks - 1 - (int)(blockIdx.x / BH);
        bh = (int)(blockIdx.x % BH);
    } else {       // neighbouring CTAs share one head's K and V in L2
        qb = (int)(blockIdx.x % n_qblocks);
        bh = (int)(blockIdx.x / n_qblocks);
    }
    const int q0 = qb * BR;
    const int dv0 = blockIdx.y * DV;
    const int dvn = min(DV, dv - dv0);
    const int b = bh / H, h = bh % H;
    const Tin *qh = q + b * st.q[0] + h * st.q[1];
    const Tin *kh = k + b * st.k[0] + h * st.k[1];
    const Tin *vh = v + b * st.v[0] + h * st.v[1];

    const int r = tid >> 3;        // query row of this thread in the block
    const int cg = tid & 7;        // lane in the row's 8-thread group
    const int row = q0 + r;

    float m = -INFINITY;           // running maximum (log2 units)
    float l = 0.f;                 // running denominator
    float acc[16];                 // columns cg*4 + 32*u + e, u < 4, e < 4
#pragma unroll
    for (int x = 0; x < 16; ++x) acc[x] = 0.f;

    const int kv_end = causal ? min(Nk, q0 + BR) : Nk;
    for (int k0 = 0; k0 < kv_end; k0 += BC) {
        // ---- S = Q_i K_j^T for this thread's 8 keys: cg + 8u
        float s[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) s[u] = 0.f;
        for (int dc = 0; dc < d; dc += DK) {
            for (int e = tid; e < BR * DK; e += NT) {
                int rr = e / DK, cc = e % DK, gr = q0 + rr, gc = dc + cc;
                Qs[rr * QS + cc] = (gr < N && gc < d) ? load_f(qh + gr * st.q[2] + gc) : 0.f;
            }
            for (int e = tid; e < BC * DK; e += NT) {
                int rr = e / DK, cc = e % DK, gr = k0 + rr, gc = dc + cc;
                Ks[rr * QS + cc] = (gr < Nk && gc < d) ? load_f(kh + gr * st.k[2] + gc) : 0.f;
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < DK; ++kk) {
                float qv = Qs[r * QS + kk];
#pragma unroll
                for (int u = 0; u < 8; ++u) s[u] = fmaf(qv, Ks[(cg + 8 * u) * QS + kk], s[u]);
            }
            __syncthreads();
        }

        // ---- online softmax update for this row
        float tmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int j = k0 + cg + 8 * u;
            bool keep = j < Nk && (!causal || j <= row);
            s[u] = keep ? s[u] * scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, s[u]);
        }
        tmax = group8_max(tmax);
        const float m_new = fmaxf(m, tmax);
        const float base = (m_new == -INFINITY) ? 0.f : m_new;  // row with no key yet
        const float alpha = exp2f(m - base);                     // 0 on the first tile
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float p = exp2f(s[u] - base);
            psum += p;
            Ps[r * PS + cg + 8 * u] = p;
        }
        psum = group8_sum(psum);
        l = l * alpha + psum;
        m = m_new;

        // ---- value tile, this CTA's columns
        for (int e = tid; e < BC * DV; e += NT) {
            int jj = e / DV, cc = e % DV, gj = k0 + jj;
            Vs[jj * DV + cc] = (gj < Nk && cc < dvn) ? load_f(vh + gj * st.v[2] + dv0 + cc) : 0.f;
        }
        __syncthreads();

        // ---- O = alpha * O + P V_j
#pragma unroll
        for (int x = 0; x < 16; ++x) acc[x] *= alpha;
#pragma unroll 4
        for (int jj = 0; jj < BC; ++jj) {
            float p = Ps[r * PS + jj];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float4 vv = *reinterpret_cast<const float4 *>(&Vs[jj * DV + cg * 4 + 32 * u]);
                acc[4 * u + 0] = fmaf(p, vv.x, acc[4 * u + 0]);
                acc[4 * u + 1] = fmaf(p, vv.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(p, vv.z, acc[4 * u + 2]);
                acc[4 * u + 3] = fmaf(p, vv.w, acc[4 * u + 3]);
            }
        }
        __syncthreads();
    }

    // ---- O / l and LSE = (m + log2 l) * ln 2
    if (row < N) {
        const float inv_l = 1.f / l;
        Tout *orow = o + b * st.o[0] + h * st.o[1] + row * st.o[2] + dv0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int c = cg * 4 + 32 * u + e;
                if (c < dvn) store_f(orow + c, acc[4 * u + e] * inv_l);
            }
        if (lse && blockIdx.y == 0 && cg == 0)
            lse[(size_t)bh * N + row] = (m + log2f(l)) * 0.69314718055994530942f;
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const Problem &p, cudaStream_t stream)
{
    auto kern = fa_general_kernel<Tin, Tout>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const int N = (int)p.N, Nk = (int)keys_of(p), d = (int)p.d, dv = (int)dv_of(p), BH = (int)(p.B * p.H);
    const int n_qblocks = (N + BR - 1) / BR;
    dim3 grid((unsigned)((int64_t)n_qblocks * BH), (unsigned)((dv + DV - 1) / DV));
    const float scale_log2 = p.scale * 1.4426950408889634f;
    Strides st;
    strides_of(p, 0, st.q);
    strides_of(p, 1, st.k);
    strides_of(p, 2, st.v);
    strides_of(p, 3, st.o);
    kern<<<grid, NT, SMEM_BYTES, stream>>>(
        static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k), static_cast<const Tin *>(p.v),
        static_cast<Tout *>(p.o), p.lse, N, Nk, d, dv, (int)p.H, n_qblocks, BH, scale_log2, p.causal, st);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_general(const Problem &p, cudaStream_t stream)
{
    const bool in_bf16 = p.in_dtype == 0, out_bf16 = p.o_dtype == 0;
    if (in_bf16 && out_bf16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(p, stream);
    if (in_bf16) return launch_typed<__nv_bfloat16, float>(p, stream);
    if (out_bf16) return launch_typed<float, __nv_bfloat16>(p, stream);
    return launch_typed<float, float>(p, stream);
}

}  // namespace fa
