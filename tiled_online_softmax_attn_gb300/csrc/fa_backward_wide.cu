// Tensor-core backward pass for wide heads: d a multiple of 128 up to 1024,
// bf16 inputs with d >= 256 and fp32 inputs (carried as bf16 hi + lo pairs,
// every product formed as hi*hi + hi*lo + lo*hi, as in the wide forward).
//
// The gradients of the forward definition by recomputation from the stored
// per-row log-sum-exp ("FlashAttention", ai360xpert.com, "Recomputation in
// the backward pass"); definitions as in fa_backward.cu:
//   P = exp(scale Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - delta) with delta_i = dO_i . O_i,  dQ = scale dS K,  dK = scale dS^T Q.
//
// A 128-row gradient tile of width d does not fit tensor memory (512 columns),
// so a CTA owns a slice of its output columns and forms the two score
// products over the whole head dimension itself, 64 columns at a time through
// a three-slot ring (as the single-CTA wide forward does):
//
// One launch, two kinds of CTA (the first n_t * d/128 of each head take the
// dK/dV role, the rest the dQ role: the two are independent, and on problems
// with few tiles neither fills the GPU alone):
//
//   dK/dV role -- 128 keys (one per tensor-memory lane) and a 128-column
//   slice of dK and dV.  Per query tile i that sees the keys:
//     S^T = K Q_i^T, dP^T = V dO_i^T              -> [0, 128), [128, 256)
//     P^T, dS^T by the elementwise warps, as bf16 (hi, lo) over their own
//       columns of S^T and dP^T
//     dV[:, slice] += P^T dO_i[:, slice]          -> [256, 384)
//     dK[:, slice] += dS^T Q_i[:, slice]          -> [384, 512)
//   dQ role -- 128 queries and a 256- (or 128-) column slice of dQ.  Per
//   key tile j the query tile sees:
//     S = Q K_j^T, dP = dO V_j^T                  -> [0, 128), [128, 256)
//     dS as bf16 (hi, lo) over the S columns
//     dQ[:, slice] += dS K_j[:, slice]            -> [256, 256 + slice)
//
// Eight elementwise warps: warp w reads tensor-memory lanes 32 (w % 4) ...
// (one row per thread) and columns 64 (w / 4) ... of the 128, and writes its
// packed bf16 results over its own fp32 columns (hi in the first 32, lo in the
// next 32), so no warp writes a column another still has to read; the MMA
// K steps address the packed operand accordingly.  Warp 8 issues the TMA
// loads, warp 9 the MMAs.  Nothing is accumulated across CTAs (no atomics;
// deterministic gradients).  Every wait is bounded as in the other kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace fa {

__device__ uint32_t g_bwdw_error_word;

namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = 128;
constexpr int EW_WARPS = 8, TMA_WARP = 8, MMA_WARP = 9, NUM_THREADS = 320;
constexpr int W = 64;                              // columns per elementwise thread
constexpr uint32_t BOX = 128 * 128;                // 128 rows x 64 bf16 (one 128-byte swizzle row each)
constexpr uint32_t STAGE = 4 * BOX;                // 64 KB
constexpr int STAGES = 3;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr int DS_KV = 128;                         // dK / dV slice width

constexpr uint32_t ERR_WAIT = 1u, ERR_DRAIN = 2u;

struct WbParams {
    int N, BH, D, n_t;     // n_t: 128-row tiles along the sequence
    int n_sl_kv;           // dK/dV slices per key tile (d / 128)
    int n_sl_q;            // dQ slices per query tile (d / dsq)
    int dsq;               // dQ slice width (256 or 128)
    float sl, scale;       // scale * log2 e, scale
    const float *lse2, *delta;  // [BH][pitch]: LSE * log2 e and delta per row
    int pitch;
    void *dq, *dk, *dv;
    int g_fp32;
    uint64_t wait_limit_ns;
};

__device__ __forceinline__ void raise_bw(volatile int *abort_flag)
{
    atomicOr(&g_bwdw_error_word, ERR_WAIT);
    *abort_flag = 1;
}

__device__ __forceinline__ void store_row32(void *base, int fp32, size_t elem, const uint32_t (&raw)[32], float mul)
{
    if (fp32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(base) + elem);
#pragma unroll
        for (int x = 0; x < 8; ++x)
            dst[x] = make_float4(__uint_as_float(raw[4 * x]) * mul, __uint_as_float(raw[4 * x + 1]) * mul,
                                 __uint_as_float(raw[4 * x + 2]) * mul, __uint_as_float(raw[4 * x + 3]) * mul);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + elem);
#pragma unroll
        for (int x = 0; x < 4; ++x)
            dst[x] = make_uint4(pack_bf16x2(__uint_as_float(raw[8 * x]) * mul, __uint_as_float(raw[8 * x + 1]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * mul, __uint_as_float(raw[8 * x + 3]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * mul, __uint_as_float(raw[8 * x + 5]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * mul, __uint_as_float(raw[8 * x + 7]) * mul));
    }
}

// Tensor-memory column of K step kk (16 values) of a packed 128-wide bf16 A
// operand: group g = kk / 4 wrote its 64 values at col0 + 64 g (hi) and
// col0 + 64 g + 32 (lo), two per column.
__device__ __forceinline__ uint32_t a_hi(uint32_t col0, int kk) { return col0 + 64u * (kk >> 2) + 8u * (kk & 3); }
__device__ __forceinline__ uint32_t a_lo(uint32_t col0, int kk) { return a_hi(col0, kk) + 32u; }

// hi = bf16(x), lo = bf16(x - hi) of two values as two packed pairs
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}

// ---------------------------------------------------------------- dK / dV
//
// Stage order per query tile (the order the MMA warp consumes): D/64 stages
// of (K, Q) column chunks for S^T, D/64 stages of (V, dO) for dP^T, one stage
// of dO[:, slice], one of Q[:, slice].  A chunk stage holds [A_hi, A_lo,
// B_hi, B_lo] boxes (A the 128-key operand), a slice stage [hi atom 0, hi
// atom 1, lo atom 0, lo atom 1] of the 128 slice columns.
template <int NPROD, bool CAUSAL>
__device__ __forceinline__ void dkdv_role(const CUtensorMap &tm_qh, const CUtensorMap &tm_ql, const CUtensorMap &tm_kh,
                                          const CUtensorMap &tm_kl, const CUtensorMap &tm_vh, const CUtensorMap &tm_vl,
                                          const CUtensorMap &tm_gh, const CUtensorMap &tm_gl, const WbParams &prm,
                                          int cta)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_b[STAGES], empty_b[STAGES], st_full, dpt_full, p_ready, ds_ready, tm_free,
        o_full, drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, D = prm.D;
    const int kt = cta / prm.n_sl_kv, sl = cta % prm.n_sl_kv;  // longest first when causal
    const int bh = (int)blockIdx.y;
    const int k0 = kt * BM, c0 = sl * DS_KV;
    const int first = CAUSAL ? kt : 0;          // query tiles before the key tile see none of its keys
    const int n_steps = prm.n_t - first;
    const int n_ch = D / 64;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty_b[s]), 1);
        }
        mbar_init(smem_addr(&st_full), 1);
        mbar_init(smem_addr(&dpt_full), 1);
        mbar_init(smem_addr(&p_ready), 32 * EW_WARPS);
        mbar_init(smem_addr(&ds_ready), 32 * EW_WARPS);
        mbar_init(smem_addr(&tm_free), 1);
        mbar_init(smem_addr(&o_full), 1);
        mbar_init(smem_addr(&drain), 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(&tmem_base_s), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint64_t limit = prm.wait_limit_ns;
    constexpr uint32_t cST = 0, cDP = 128, cDV = 256, cDK = 384;

    if (warp == TMA_WARP) {
        // ================================================================ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int it = 0;
            bool ok = true;
            auto acquire = [&](uint32_t bytes) -> int {
                const int st = it % STAGES;
                if (!wait_or_abort(smem_addr(&empty_b[st]), (uint32_t)(((it / STAGES) & 1) ^ 1), limit, &abort_flag))
                    return -1;
                mbar_arrive_expect_tx(smem_addr(&full_b[st]), bytes);
                return st;
            };
            auto chunks = [&](const void *ah, const void *al, const void *bh_, const void *bl, int a_row, int b_row) {
                for (int c = 0; ok && c < n_ch; ++c) {
                    const int st = acquire(NPROD == 3 ? 4 * BOX : 2 * BOX);
                    if (st < 0) { ok = false; return; }
                    const uint32_t dst = s_base + st * STAGE, fb = smem_addr(&full_b[st]);
                    tma_load_3d(dst, ah, fb, c * 64, a_row, bh, pol);
                    tma_load_3d(dst + 2 * BOX, bh_, fb, c * 64, b_row, bh, pol);
                    if (NPROD == 3) {
                        tma_load_3d(dst + BOX, al, fb, c * 64, a_row, bh, pol);
                        tma_load_3d(dst + 3 * BOX, bl, fb, c * 64, b_row, bh, pol);
                    }
                    ++it;
                }
            };
            auto slice = [&](const void *th, const void *tl, int row) {
                const int st = acquire(NPROD == 3 ? 4 * BOX : 2 * BOX);
                if (st < 0) { ok = false; return; }
                const uint32_t dst = s_base + st * STAGE, fb = smem_addr(&full_b[st]);
                for (int a = 0; a < 2; ++a) {
                    tma_load_3d(dst + a * BOX, th, fb, c0 + a * 64, row, bh, pol);
                    if (NPROD == 3) tma_load_3d(dst + (2 + a) * BOX, tl, fb, c0 + a * 64, row, bh, pol);
                }
                ++it;
            };
            for (int s = 0; ok && s < n_steps; ++s) {
                const int q0 = (first + s) * BM;
                chunks(&tm_kh, &tm_kl, &tm_qh, &tm_ql, k0, q0);
                chunks(&tm_vh, &tm_vl, &tm_gh, &tm_gl, k0, q0);
                if (ok) slice(&tm_gh, &tm_gl, q0);
                if (ok) slice(&tm_qh, &tm_ql, q0);
            }
            if (!ok) {
                if (!abort_flag) raise_bw(&abort_flag);
                for (int j = max(0, it - STAGES); j < it; ++j)
                    if (!mbar_wait_bounded(smem_addr(&full_b[j % STAGES]), (uint32_t)((j / STAGES) & 1), limit))
                        atomicOr(&g_bwdw_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================================================================ MMA issuer
        {
            const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0);       // A and B K-major
            const uint32_t id_g = idesc_bf16_f32(BM, DS_KV, 0, 1);    // B (dO or Q slice) MN-major
            int it = 0;
            bool ok = true, issued = false;
            auto wait_full = [&]() -> int {
                const int st = it % STAGES;
                if (!wait_or_abort_w(smem_addr(&full_b[st]), (uint32_t)((it / STAGES) & 1), limit, &abort_flag))
                    return -1;
                tc_fence_after();
                return st;
            };
            // d[tmem] = A B^T over the whole head dimension, chunk by chunk
            auto score = [&](uint32_t d) -> bool {
                for (int c = 0; c < n_ch; ++c) {
                    const int st = wait_full();
                    if (st < 0) return false;
                    const uint32_t base = s_base + st * STAGE;
                    const uint64_t ah = sdesc_sw128(base, 16, 1024), al = sdesc_sw128(base + BOX, 16, 1024);
                    const uint64_t bh_ = sdesc_sw128(base + 2 * BOX, 16, 1024), bl = sdesc_sw128(base + 3 * BOX, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t off = (uint64_t)(kk * 2);  // 32 bytes along K
                        mma_ss_w(d, ah + off, bh_ + off, id_s, (c > 0 || kk > 0) ? 1u : 0u);
                        if (NPROD == 3) {
                            mma_ss_w(d, ah + off, bl + off, id_s, 1u);
                            mma_ss_w(d, al + off, bh_ + off, id_s, 1u);
                        }
                    }
                    issued = true;
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
                return true;
            };
            // acc[tmem] += X^T B_slice, X packed in tensor memory at col0 (hi, lo)
            auto grad = [&](uint32_t acc, uint32_t col0, bool first_step) -> bool {
                const int st = wait_full();
                if (st < 0) return false;
                const uint32_t base = s_base + st * STAGE;
                const uint64_t gh = sdesc_sw128(base, BOX, 1024), gl = sdesc_sw128(base + 2 * BOX, BOX, 1024);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = (uint64_t)((kk * 16 * 128) >> 4);
                    mma_ts_w(acc, tmem + a_hi(col0, kk), gh + off, id_g, (!first_step || kk > 0) ? 1u : 0u);
                    if (NPROD == 3) {
                        mma_ts_w(acc, tmem + a_lo(col0, kk), gh + off, id_g, 1u);
                        mma_ts_w(acc, tmem + a_hi(col0, kk), gl + off, id_g, 1u);
                    }
                }
                issued = true;
                mma_commit_w(smem_addr(&empty_b[st]));
                ++it;
                return true;
            };
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s > 0 && !wait_or_abort_w(smem_addr(&tm_free), (uint32_t)((s - 1) & 1), limit, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (!score(tmem + cST)) { ok = false; break; }
                mma_commit_w(smem_addr(&st_full));
                if (!score(tmem + cDP)) { ok = false; break; }
                mma_commit_w(smem_addr(&dpt_full));
                if (!wait_or_abort_w(smem_addr(&p_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (!grad(tmem + cDV, cST, s == 0)) { ok = false; break; }
                if (!wait_or_abort_w(smem_addr(&ds_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (!grad(tmem + cDK, cDP, s == 0)) { ok = false; break; }
                mma_commit_w(smem_addr(&tm_free));
            }
            if (ok) {
                mma_commit_w(smem_addr(&o_full));
            } else {
                if (!abort_flag) raise_bw(&abort_flag);
                if (issued) {
                    mma_commit_w(smem_addr(&drain));
                    if (!mbar_wait_bounded(smem_addr(&drain), 0, limit)) atomicOr(&g_bwdw_error_word, ERR_DRAIN);
                }
            }
        }
        __syncwarp();
    } else {
        // ================================================================ elementwise + epilogue
        const int qw = warp & 3, g = warp >> 2;     // lane quarter, column half
        const int kj = k0 + qw * 32 + lane;         // this thread's key
        const uint32_t lb = tmem + ((uint32_t)(qw * 32) << 16);
        const float sl = prm.sl;
        bool ok = true;
        auto uwait = [&](const uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(smem_addr(bar), parity, limit, &abort_flag));
        };
        for (int s = 0; ok && s < n_steps; ++s) {
            const int qt0 = (first + s) * BM, q0 = qt0 + g * W;  // this thread's 64 queries start at q0
            const bool masked = k0 + BM > N || qt0 + BM > N || (CAUSAL && qt0 < k0 + BM);
            const float *l2v = prm.lse2 + (size_t)bh * prm.pitch + q0;
            const float *dev = prm.delta + (size_t)bh * prm.pitch + q0;
            if (!uwait(&st_full, (uint32_t)(s & 1))) { ok = false; break; }
            tc_fence_after();
            // ---- P^T: weights of this key for the 64 queries, hi (and lo) over its S^T columns
            uint32_t ph[W / 2], pl[W / 2];
            {
                uint32_t raw[W];
                tmem_ld64(lb + cST + g * W, raw);
                const uint64_t sl2 = f2_pack(sl, sl);
#pragma unroll
                for (int c4 = 0; c4 < W / 4; ++c4) {
                    const float4 l4 = __ldg(reinterpret_cast<const float4 *>(l2v) + c4);
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int c = 4 * c4 + e;
                        const uint64_t nl = e ? f2_pack(-l4.z, -l4.w) : f2_pack(-l4.x, -l4.y);
                        float a0, a1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), sl2, nl), a0, a1);
                        float w0 = ex2(a0), w1 = ex2(a1);
                        if (masked) {  // the padded LSE entries past N are never used unmasked
                            const int q = q0 + c;
                            w0 = (kj < N && q < N && (!CAUSAL || kj <= q)) ? w0 : 0.f;
                            w1 = (kj < N && q + 1 < N && (!CAUSAL || kj <= q + 1)) ? w1 : 0.f;
                        }
                        if (NPROD == 3) split2(w0, w1, ph[c / 2], pl[c / 2]);
                        else ph[c / 2] = pack_bf16x2(w0, w1);
                    }
                }
            }
            {
                uint32_t h32[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) h32[c] = ph[c];
                tmem_st32(lb + cST + g * W, h32);
                if (NPROD == 3) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) h32[c] = pl[c];
                    tmem_st32(lb + cST + g * W + 32, h32);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(&p_ready));
            // ---- dS^T = P^T (dP^T - delta), hi (and lo) over its dP^T columns
            if (!uwait(&dpt_full, (uint32_t)(s & 1))) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t raw[W];
                tmem_ld64(lb + cDP + g * W, raw);
                uint32_t dh[W / 2], dl[W / 2];
#pragma unroll
                for (int c4 = 0; c4 < W / 4; ++c4) {
                    const float4 d4 = __ldg(reinterpret_cast<const float4 *>(dev) + c4);
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int c = 4 * c4 + e;
                        // the weights the dV product uses: hi (+ lo)
                        float p0 = __uint_as_float(ph[c / 2] << 16), p1 = __uint_as_float(ph[c / 2] & 0xFFFF0000u);
                        if (NPROD == 3) {
                            p0 += __uint_as_float(pl[c / 2] << 16);
                            p1 += __uint_as_float(pl[c / 2] & 0xFFFF0000u);
                        }
                        const uint64_t nd = e ? f2_pack(-d4.z, -d4.w) : f2_pack(-d4.x, -d4.y);
                        const uint64_t t = f2_add(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), nd);
                        float d0, d1;
                        f2_unpack(f2_mul(f2_pack(p0, p1), t), d0, d1);
                        if (masked) {  // a masked weight is exactly 0 and its dP may be anything
                            d0 = p0 != 0.f ? d0 : 0.f;
                            d1 = p1 != 0.f ? d1 : 0.f;
                        }
                        if (NPROD == 3) split2(d0, d1, dh[c / 2], dl[c / 2]);
                        else dh[c / 2] = pack_bf16x2(d0, d1);
                    }
                }
                tmem_st32(lb + cDP + g * W, dh);
                if (NPROD == 3) tmem_st32(lb + cDP + g * W + 32, dl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(&ds_ready));
        }
        if (ok && uwait(&o_full, 0)) {
            tc_fence_after();
            const size_t row = ((size_t)bh * N + kj) * D + c0;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {  // this warp's two 32-column chunks of the slice
                const int col = g * W + c * 32;
                uint32_t raw[32];
                tmem_ld32(lb + cDV + col, raw);
                if (kj < N) store_row32(prm.dv, prm.g_fp32, row + col, raw, 1.f);
                tmem_ld32(lb + cDK + col, raw);
                if (kj < N) store_row32(prm.dk, prm.g_fp32, row + col, raw, prm.scale);
            }
        } else if (!abort_flag) {
            raise_bw(&abort_flag);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- dQ
//
// Stage order per key tile: D/64 stages of (Q, K) chunks for S, D/64 of
// (dO, V) for dP, then the K slice: DSQ / 64 atoms of hi in one stage and of
// lo in the next (fp32 inputs).
template <int NPROD, int DSQ, bool CAUSAL>
__device__ __forceinline__ void dq_role(const CUtensorMap &tm_qh, const CUtensorMap &tm_ql, const CUtensorMap &tm_kh,
                                        const CUtensorMap &tm_kl, const CUtensorMap &tm_vh, const CUtensorMap &tm_vl,
                                        const CUtensorMap &tm_gh, const CUtensorMap &tm_gl, const WbParams &prm, int cta)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_b[STAGES], empty_b[STAGES], s_full, dp_full, ds_ready, tm_free, o_full, drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, D = prm.D;
    const int qi = cta / prm.n_sl_q, sl = cta % prm.n_sl_q;
    const int qt = CAUSAL ? prm.n_t - 1 - qi : qi;  // longest first when causal
    const int bh = (int)blockIdx.y;
    const int q0 = qt * BM, c0 = sl * DSQ;
    const int n_steps = CAUSAL ? qt + 1 : prm.n_t;  // key tiles this query tile sees
    const int n_ch = D / 64;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty_b[s]), 1);
        }
        mbar_init(smem_addr(&s_full), 1);
        mbar_init(smem_addr(&dp_full), 1);
        mbar_init(smem_addr(&ds_ready), 32 * EW_WARPS);
        mbar_init(smem_addr(&tm_free), 1);
        mbar_init(smem_addr(&o_full), 1);
        mbar_init(smem_addr(&drain), 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(&tmem_base_s), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint64_t limit = prm.wait_limit_ns;
    constexpr uint32_t cS = 0, cDP = 128, cDQ = 256;
    constexpr int NA = DSQ / 64;  // 64-column atoms of the K slice

    if (warp == TMA_WARP) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int it = 0;
            bool ok = true;
            auto acquire = [&](uint32_t bytes) -> int {
                const int st = it % STAGES;
                if (!wait_or_abort(smem_addr(&empty_b[st]), (uint32_t)(((it / STAGES) & 1) ^ 1), limit, &abort_flag))
                    return -1;
                mbar_arrive_expect_tx(smem_addr(&full_b[st]), bytes);
                return st;
            };
            auto chunks = [&](const void *ah, const void *al, const void *bh_, const void *bl, int a_row, int b_row) {
                for (int c = 0; ok && c < n_ch; ++c) {
                    const int st = acquire(NPROD == 3 ? 4 * BOX : 2 * BOX);
                    if (st < 0) { ok = false; return; }
                    const uint32_t dst = s_base + st * STAGE, fb = smem_addr(&full_b[st]);
                    tma_load_3d(dst, ah, fb, c * 64, a_row, bh, pol);
                    tma_load_3d(dst + 2 * BOX, bh_, fb, c * 64, b_row, bh, pol);
                    if (NPROD == 3) {
                        tma_load_3d(dst + BOX, al, fb, c * 64, a_row, bh, pol);
                        tma_load_3d(dst + 3 * BOX, bl, fb, c * 64, b_row, bh, pol);
                    }
                    ++it;
                }
            };
            for (int s = 0; ok && s < n_steps; ++s) {
                const int kr = s * BM;
                chunks(&tm_qh, &tm_ql, &tm_kh, &tm_kl, q0, kr);
                chunks(&tm_gh, &tm_gl, &tm_vh, &tm_vl, q0, kr);
                for (int part = 0; ok && part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = acquire(NA * BOX);
                    if (st < 0) { ok = false; break; }
                    const uint32_t dst = s_base + st * STAGE, fb = smem_addr(&full_b[st]);
                    for (int a = 0; a < NA; ++a)
                        tma_load_3d(dst + a * BOX, part ? &tm_kl : &tm_kh, fb, c0 + a * 64, kr, bh, pol);
                    ++it;
                }
            }
            if (!ok) {
                if (!abort_flag) raise_bw(&abort_flag);
                for (int j = max(0, it - STAGES); j < it; ++j)
                    if (!mbar_wait_bounded(smem_addr(&full_b[j % STAGES]), (uint32_t)((j / STAGES) & 1), limit))
                        atomicOr(&g_bwdw_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        {
            const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0);
            const uint32_t id_g = idesc_bf16_f32(BM, DSQ, 0, 1);
            int it = 0;
            bool ok = true, issued = false;
            auto wait_full = [&]() -> int {
                const int st = it % STAGES;
                if (!wait_or_abort_w(smem_addr(&full_b[st]), (uint32_t)((it / STAGES) & 1), limit, &abort_flag))
                    return -1;
                tc_fence_after();
                return st;
            };
            auto score = [&](uint32_t d) -> bool {
                for (int c = 0; c < n_ch; ++c) {
                    const int st = wait_full();
                    if (st < 0) return false;
                    const uint32_t base = s_base + st * STAGE;
                    const uint64_t ah = sdesc_sw128(base, 16, 1024), al = sdesc_sw128(base + BOX, 16, 1024);
                    const uint64_t bh_ = sdesc_sw128(base + 2 * BOX, 16, 1024), bl = sdesc_sw128(base + 3 * BOX, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t off = (uint64_t)(kk * 2);
                        mma_ss_w(d, ah + off, bh_ + off, id_s, (c > 0 || kk > 0) ? 1u : 0u);
                        if (NPROD == 3) {
                            mma_ss_w(d, ah + off, bl + off, id_s, 1u);
                            mma_ss_w(d, al + off, bh_ + off, id_s, 1u);
                        }
                    }
                    issued = true;
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
                return true;
            };
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s > 0 && !wait_or_abort_w(smem_addr(&tm_free), (uint32_t)((s - 1) & 1), limit, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (!score(tmem + cS)) { ok = false; break; }
                mma_commit_w(smem_addr(&s_full));
                if (!score(tmem + cDP)) { ok = false; break; }
                mma_commit_w(smem_addr(&dp_full));
                if (!wait_or_abort_w(smem_addr(&ds_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                // dQ[:, slice] += dS K_slice: dS packed over the S columns
                for (int part = 0; ok && part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = wait_full();
                    if (st < 0) { ok = false; break; }
                    const uint64_t kd = sdesc_sw128(s_base + st * STAGE, BOX, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk) {
                        const uint64_t off = (uint64_t)((kk * 16 * 128) >> 4);
                        if (part == 0) {
                            mma_ts_w(tmem + cDQ, tmem + a_hi(cS, kk), kd + off, id_g, (s > 0 || kk > 0) ? 1u : 0u);
                            if (NPROD == 3) mma_ts_w(tmem + cDQ, tmem + a_lo(cS, kk), kd + off, id_g, 1u);
                        } else {
                            mma_ts_w(tmem + cDQ, tmem + a_hi(cS, kk), kd + off, id_g, 1u);
                        }
                    }
                    issued = true;
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
                if (!ok) break;
                mma_commit_w(smem_addr(&tm_free));
            }
            if (ok) {
                mma_commit_w(smem_addr(&o_full));
            } else {
                if (!abort_flag) raise_bw(&abort_flag);
                if (issued) {
                    mma_commit_w(smem_addr(&drain));
                    if (!mbar_wait_bounded(smem_addr(&drain), 0, limit)) atomicOr(&g_bwdw_error_word, ERR_DRAIN);
                }
            }
        }
        __syncwarp();
    } else {
        const int qw = warp & 3, g = warp >> 2;
        const int qi = q0 + qw * 32 + lane;         // this thread's query
        const uint32_t lb = tmem + ((uint32_t)(qw * 32) << 16);
        const float sl = prm.sl;
        const float l2 = qi < N ? prm.lse2[(size_t)bh * prm.pitch + qi] : 0.f;
        const float de = qi < N ? prm.delta[(size_t)bh * prm.pitch + qi] : 0.f;
        bool ok = true;
        auto uwait = [&](const uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(smem_addr(bar), parity, limit, &abort_flag));
        };
        for (int s = 0; ok && s < n_steps; ++s) {
            const int kt0 = s * BM, kb = kt0 + g * W;   // this thread's 64 keys start at kb
            const bool masked = kt0 + BM > N || q0 + BM > N || (CAUSAL && kt0 + BM > q0);
            if (!uwait(&s_full, (uint32_t)(s & 1))) { ok = false; break; }
            tc_fence_after();
            float p[W];
            {
                uint32_t raw[W];
                tmem_ld64(lb + cS + g * W, raw);
                const uint64_t sl2 = f2_pack(sl, sl), nl = f2_pack(-l2, -l2);
#pragma unroll
                for (int c = 0; c < W; c += 2) {
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), sl2, nl), a0, a1);
                    float w0 = ex2(a0), w1 = ex2(a1);
                    if (masked) {
                        const int k = kb + c;
                        w0 = (qi < N && k < N && (!CAUSAL || k <= qi)) ? w0 : 0.f;
                        w1 = (qi < N && k + 1 < N && (!CAUSAL || k + 1 <= qi)) ? w1 : 0.f;
                    }
                    if (NPROD == 1) {  // the bf16 weights, as the dK/dV kernel uses them
                        const uint32_t h = pack_bf16x2(w0, w1);
                        w0 = __uint_as_float(h << 16);
                        w1 = __uint_as_float(h & 0xFFFF0000u);
                    }
                    p[c] = w0;
                    p[c + 1] = w1;
                }
            }
            if (!uwait(&dp_full, (uint32_t)(s & 1))) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t raw[W];
                tmem_ld64(lb + cDP + g * W, raw);
                uint32_t dh[W / 2], dl[W / 2];
                const uint64_t nd = f2_pack(-de, -de);
#pragma unroll
                for (int c = 0; c < W; c += 2) {
                    const uint64_t t = f2_add(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), nd);
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]), t), d0, d1);
                    if (masked) {
                        d0 = p[c] != 0.f ? d0 : 0.f;
                        d1 = p[c + 1] != 0.f ? d1 : 0.f;
                    }
                    if (NPROD == 3) split2(d0, d1, dh[c / 2], dl[c / 2]);
                    else dh[c / 2] = pack_bf16x2(d0, d1);
                }
                // over this group's own S columns (read above)
                tmem_st32(lb + cS + g * W, dh);
                if (NPROD == 3) tmem_st32(lb + cS + g * W + 32, dl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(&ds_ready));
        }
        if (ok && uwait(&o_full, 0)) {
            tc_fence_after();
            const size_t row = ((size_t)bh * N + qi) * D + c0;
#pragma unroll 1
            for (int c = g * (DSQ / 2); c < (g + 1) * (DSQ / 2); c += 32) {
                uint32_t raw[32];
                tmem_ld32(lb + cDQ + c, raw);
                if (qi < N) store_row32(prm.dq, prm.g_fp32, row + c, raw, prm.scale);
            }
        } else if (!abort_flag) {
            raise_bw(&abort_flag);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// One launch for both: the first n_t * n_sl_kv CTAs (of each head) take the
// dK/dV role, the rest the dQ role.  The two are independent, and on problems
// with few tiles neither fills the GPU alone.
template <int NPROD, int DSQ, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fa_bwdw_kernel(const __grid_constant__ CUtensorMap tm_qh, const __grid_constant__ CUtensorMap tm_ql,
               const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_kl,
               const __grid_constant__ CUtensorMap tm_vh, const __grid_constant__ CUtensorMap tm_vl,
               const __grid_constant__ CUtensorMap tm_gh, const __grid_constant__ CUtensorMap tm_gl, const WbParams prm)
{
    const int n_kv = prm.n_t * prm.n_sl_kv;
    if ((int)blockIdx.x < n_kv)
        dkdv_role<NPROD, CAUSAL>(tm_qh, tm_ql, tm_kh, tm_kl, tm_vh, tm_vl, tm_gh, tm_gl, prm, (int)blockIdx.x);
    else
        dq_role<NPROD, DSQ, CAUSAL>(tm_qh, tm_ql, tm_kh, tm_kl, tm_vh, tm_vl, tm_gh, tm_gl, prm, (int)blockIdx.x - n_kv);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [BH, N, d] bf16, box 64 columns x 128 rows, 128-byte swizzle; rows past N read as zeros.
bool make_map(CUtensorMap *map, const void *ptr, int64_t BH, int64_t N, int64_t d)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)(N * d * 2)};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool backward_wide_supported(const BackwardProblem &p)
{
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    const bool fp32_in = p.in_dtype == 1;
    return p.d % 128 == 0 && p.d <= 1024 && (fp32_in ? p.d >= 128 : p.d >= 256) && p.scale > 0.f &&
           p.B * p.H <= 65535 && al16(p.q) && al16(p.k) && al16(p.v) && al16(p.dout) && al16(p.dq) && al16(p.dk) &&
           al16(p.dv);
}

size_t backward_wide_copy_bytes(const BackwardProblem &p)
{
    if (p.in_dtype != 1) return 0;
    return 8 * al256((size_t)(p.B * p.H * p.N * p.d) * 2);  // Q, K, V, dO as bf16 hi and lo
}

cudaError_t launch_backward_wide(const BackwardProblem &p, void *workspace, cudaStream_t stream, const char **detail)
{
    const int64_t BH = p.B * p.H;
    const int pitch = (int)((p.N + 127) / 128 * 128);
    float *delta = nullptr, *lse2 = nullptr;
    cudaError_t e = launch_backward_delta(p, workspace, stream, pitch, &delta, &lse2);
    if (e != cudaSuccess) return e;
    const int nprod = p.in_dtype == 1 ? 3 : 1;
    const void *src[4] = {p.q, p.k, p.v, p.dout};
    const void *hi[4] = {p.q, p.k, p.v, p.dout}, *lo[4] = {p.q, p.k, p.v, p.dout};
    if (nprod == 3) {
        uint8_t *c = static_cast<uint8_t *>(workspace) + backward_workspace_bytes(p);
        const size_t n = (size_t)(BH * p.N * p.d), one = al256(n * 2);
        void *h[4], *l[4];
        for (int t = 0; t < 4; ++t) {
            h[t] = c + (2 * t) * one;
            l[t] = c + (2 * t + 1) * one;
            hi[t] = h[t];
            lo[t] = l[t];
        }
        if ((e = launch_split_hilo(reinterpret_cast<const float *const *>(src), h, l, 4, n, stream)) != cudaSuccess)
            return e;
    }
    CUtensorMap m[8];
    for (int t = 0; t < 4; ++t)
        if (!make_map(&m[2 * t], hi[t], BH, p.N, p.d) || !make_map(&m[2 * t + 1], lo[t], BH, p.N, p.d)) {
            *detail = "cuTensorMapEncodeTiled failed or is unavailable";
            return cudaErrorInvalidValue;
        }
    WbParams prm{};
    prm.N = (int)p.N;
    prm.BH = (int)BH;
    prm.D = (int)p.d;
    prm.n_t = (int)((p.N + BM - 1) / BM);
    prm.sl = p.scale * 1.4426950408889634f;
    prm.scale = p.scale;
    prm.lse2 = lse2;
    prm.delta = delta;
    prm.pitch = pitch;
    prm.dq = p.dq;
    prm.dk = p.dk;
    prm.dv = p.dv;
    prm.g_fp32 = p.grad_dtype == 1;
    prm.wait_limit_ns = 2000000000ull;
    // maps: Q, K, V, dO (hi, lo each) as the kernel takes them
    const bool wide_q = p.d % 256 == 0;
    prm.dsq = wide_q ? 256 : 128;
    prm.n_sl_kv = (int)(p.d / DS_KV);
    prm.n_sl_q = (int)(p.d / prm.dsq);
    const unsigned gx = (unsigned)(prm.n_t * (prm.n_sl_kv + prm.n_sl_q));
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        kern<<<dim3(gx, (unsigned)BH), NUM_THREADS, SMEM_BYTES, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                                                                          prm);
        return cudaGetLastError();
    };
    if (nprod == 3) {
        if (wide_q) return p.causal ? go(fa_bwdw_kernel<3, 256, true>) : go(fa_bwdw_kernel<3, 256, false>);
        return p.causal ? go(fa_bwdw_kernel<3, 128, true>) : go(fa_bwdw_kernel<3, 128, false>);
    }
    if (wide_q) return p.causal ? go(fa_bwdw_kernel<1, 256, true>) : go(fa_bwdw_kernel<1, 256, false>);
    return p.causal ? go(fa_bwdw_kernel<1, 128, true>) : go(fa_bwdw_kernel<1, 128, false>);
}

cudaError_t bwdw_error_word_ptr(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_bwdw_error_word);
}

}  // namespace fa
