// Wide-head attention forward on the tensor cores: head dimensions 128..1024
// (multiples of 128) with fp32 inputs, and 256..1024 with bf16 inputs.
//
// Same algorithm as the main tensor-core kernel -- the tiled online-softmax
// forward of "Deep Learning - Flash Attention" ("An Example", steps 4-7) and
// "The Details of Flash Attention" ("Tiling the Loop"), unnormalised O with
// lazy rescaling, one division at the end -- organised for heads too wide
// for a 128-row O tile to live in tensor memory:
//
//   * a CTA owns one 128-row query tile, one 256- (or 128-) column slice of O
//     and a contiguous range of key tiles (a "split");
//   * S = Q K^T is accumulated over the whole head dimension in 64-column
//     chunks streamed through a three-slot shared-memory ring (each O slice
//     recomputes S: the price of keeping O in tensor memory);
//   * fp32 inputs are carried as two bf16 terms, x = hi + lo with
//     hi = bf16(x), lo = bf16(x - hi) (a pre-pass writes them to the
//     workspace), and every product is formed as hi*hi + hi*lo + lo*hi with
//     fp32 accumulation: about 16 significant bits per operand, so the
//     dropped lo*lo term is ~2^-16 of each product.  P is split the same way;
//   * when one split per query tile leaves SMs idle, the key range is cut
//     into several splits whose partial (O, m, l) go to the workspace and a
//     combine kernel merges them with the rule of "FlashAttention Engine:
//     Hardware-Aware Exact Attention & SRAM Tiling" ("Core FlashAttention
//     Mechanics", item 3):  m = max_s m_s,  l = sum_s l_s 2^(m_s - m),
//     O = sum_s O_s 2^(m_s - m) / l.
//
// Warps: 0-3 softmax and epilogue (one query row per thread), 4 TMA
// producer, 5 MMA issuer.  Tensor memory: S / P at columns [0, 128)
// (P_hi over [0, 64), P_lo over [64, 128)), O slice at [256, 256 + DV).
// Every wait is bounded as in the main kernel.
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

__device__ uint32_t g_wide_error_word;

namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int NUM_THREADS = 192;
constexpr int TMA_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr int STAGES = 3;
constexpr uint32_t STAGE_BYTES = 65536;
constexpr uint32_t BOX_BYTES = BM * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle atom row each)
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 256;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int MAX_SPLITS = 16;

constexpr uint32_t ERR_WAIT = 16u;   // bits distinct from the main kernel's
constexpr uint32_t ERR_DRAIN = 32u;

struct WideParams {
    int N, BH, D;
    int n_q, n_dv, n_split, tiles_per_split, n_kv;
    float scale_log2;
    uint64_t wait_limit_ns;
    int direct;        // 1: O normalised into `o` and LSE; 0: partials into the workspace
    void *o;
    int o_fp32;
    float *lse;
    float *o_part;     // [n_split][BH][N][D], unnormalised
    float *m_part;     // [n_split][BH][N], reference maximum (log2 units), -inf if empty
    float *l_part;     // [n_split][BH][N], exact denominator
    float *d_part;     // [n_split][BH][N], bf16 rounding of the top weights (bf16 inputs)
};

__device__ __forceinline__ void raise_wide(uint32_t bit, volatile int *abort_flag)
{
    atomicOr(&g_wide_error_word, bit);
    *abort_flag = 1;
}

template <int NPROD, int DV, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fa_wide_kernel(const __grid_constant__ CUtensorMap tm_qh, const __grid_constant__ CUtensorMap tm_ql,
               const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_kl,
               const __grid_constant__ CUtensorMap tm_vh, const __grid_constant__ CUtensorMap tm_vl,
               const WideParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_b[STAGES], empty_b[STAGES], s_full, p_full, o_full, drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, D = prm.D;
    const int per_q = prm.n_dv * prm.n_split;
    const int qt = CAUSAL ? prm.n_q - 1 - (int)(blockIdx.x / per_q) : (int)(blockIdx.x / per_q);
    const int rem = (int)(blockIdx.x % per_q);
    const int dvc = rem / prm.n_split, sp = rem % prm.n_split;
    const int bh = (int)blockIdx.y;
    const int q0 = qt * BM, dv0 = dvc * DV;
    const int kv_need = CAUSAL ? min(prm.n_kv, qt + 1) : prm.n_kv;
    const int kv_lo = sp * prm.tiles_per_split;
    const int n_j = min(kv_lo + prm.tiles_per_split, kv_need) - kv_lo;
    const size_t part_row = ((size_t)sp * prm.BH + bh) * N;  // row base of this split's partials

    if (n_j <= 0) {  // a split with no visible key (causal): an empty partial
        if (!prm.direct && dvc == 0 && warp < 4) {
            const int grow = q0 + (int)threadIdx.x;
            if (grow < N) {
                prm.m_part[part_row + grow] = -INFINITY;
                prm.l_part[part_row + grow] = 0.f;
                prm.d_part[part_row + grow] = 0.f;
            }
        }
        return;
    }

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    const int n_sc = D / 64;  // 64-column chunks of the score product

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty_b[s]), 1);
        }
        mbar_init(smem_addr(&s_full), 1);
        mbar_init(smem_addr(&p_full), 128);
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
            for (int jj = 0; ok && jj < n_j; ++jj) {
                const int k0 = (kv_lo + jj) * BN;
                for (int c = 0; ok && c < n_sc; ++c) {
                    const int st = acquire(NPROD == 3 ? 4 * BOX_BYTES : 2 * BOX_BYTES);
                    if (st < 0) { ok = false; break; }
                    const uint32_t dst = s_base + st * STAGE_BYTES, fb = smem_addr(&full_b[st]);
                    tma_load_3d(dst, &tm_qh, fb, c * 64, q0, bh, pol);
                    tma_load_3d(dst + 2 * BOX_BYTES, &tm_kh, fb, c * 64, k0, bh, pol);
                    if (NPROD == 3) {
                        tma_load_3d(dst + BOX_BYTES, &tm_ql, fb, c * 64, q0, bh, pol);
                        tma_load_3d(dst + 3 * BOX_BYTES, &tm_kl, fb, c * 64, k0, bh, pol);
                    }
                    ++it;
                }
                for (int part = 0; ok && part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = acquire((DV / 64) * BOX_BYTES);
                    if (st < 0) { ok = false; break; }
                    const uint32_t dst = s_base + st * STAGE_BYTES, fb = smem_addr(&full_b[st]);
                    for (int a = 0; a < DV / 64; ++a)
                        tma_load_3d(dst + a * BOX_BYTES, part ? &tm_vl : &tm_vh, fb, dv0 + a * 64, k0, bh, pol);
                    ++it;
                }
            }
            if (!ok) {
                if (!abort_flag) raise_wide(ERR_WAIT, &abort_flag);
                // every issued load must land before the CTA exits
                for (int j = max(0, it - STAGES); j < it; ++j)
                    if (!mbar_wait_bounded(smem_addr(&full_b[j % STAGES]), (uint32_t)((j / STAGES) & 1), limit))
                        atomicOr(&g_wide_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================================================================ MMA issuer
        {  // whole warp, converged; elect.sync picks the issuing lane
            const uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(BM, DV, 0, 1);
            const uint32_t tS = tmem, tO = tmem + COL_O;
            int it = 0;
            bool ok = true, issued = false;
            auto wait_full = [&]() -> int {
                const int st = it % STAGES;
                if (!wait_or_abort_w(smem_addr(&full_b[st]), (uint32_t)((it / STAGES) & 1), limit, &abort_flag))
                    return -1;
                tc_fence_after();
                return st;
            };
            for (int jj = 0; ok && jj < n_j; ++jj) {
                for (int c = 0; c < n_sc; ++c) {
                    const int st = wait_full();
                    if (st < 0) { ok = false; break; }
                    const uint32_t base = s_base + st * STAGE_BYTES;
                    const uint64_t dqh = sdesc_sw128(base, 16, 1024), dql = sdesc_sw128(base + BOX_BYTES, 16, 1024);
                    const uint64_t dkh = sdesc_sw128(base + 2 * BOX_BYTES, 16, 1024),
                                   dkl = sdesc_sw128(base + 3 * BOX_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t off = (uint64_t)(kk * 2);  // 32 bytes along K
                        mma_ss_w(tS, dqh + off, dkh + off, idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
                        if (NPROD == 3) {
                            mma_ss_w(tS, dqh + off, dkl + off, idesc_s, 1u);
                            mma_ss_w(tS, dql + off, dkh + off, idesc_s, 1u);
                        }
                    }
                    issued = true;
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
                if (!ok) break;
                mma_commit_w(smem_addr(&s_full));
                if (!wait_or_abort_w(smem_addr(&p_full), (uint32_t)(jj & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int part = 0; part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = wait_full();
                    if (st < 0) { ok = false; break; }
                    const uint64_t dv = sdesc_sw128(s_base + st * STAGE_BYTES, BOX_BYTES, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t voff = (uint64_t)((kk * 16 * 128) >> 4);
                        if (part == 0) {
                            mma_ts_w(tO, tS + kk * 8, dv + voff, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                            if (NPROD == 3) mma_ts_w(tO, tS + 64 + kk * 8, dv + voff, idesc_o, 1u);
                        } else {
                            mma_ts_w(tO, tS + kk * 8, dv + voff, idesc_o, 1u);
                        }
                    }
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
            }
            if (ok) {
                mma_commit_w(smem_addr(&o_full));
            } else {
                if (!abort_flag) raise_wide(ERR_WAIT, &abort_flag);
                if (issued) {
                    mma_commit_w(smem_addr(&drain));
                    if (!mbar_wait_bounded(smem_addr(&drain), 0, limit)) atomicOr(&g_wide_error_word, ERR_DRAIN);
                }
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax + epilogue
        const int r = warp * 32 + lane;
        const int grow = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t tS = lane_base, tO = lane_base + COL_O;
        const float sl = prm.scale_log2;
        float m = -INFINITY, l = 0.f, dq = 0.f;
        bool ok = true;
        for (int jj = 0; jj < n_j; ++jj) {
            if (!wait_or_abort(smem_addr(&s_full), (uint32_t)(jj & 1), limit, &abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[BN];
            {
                uint32_t raw[BN];
                tmem_ld128(tS, raw);
#pragma unroll
                for (int x = 0; x < BN; ++x) s[x] = __uint_as_float(raw[x]);
            }
            const int kc0 = (kv_lo + jj) * BN;
            int lim = N - kc0;
            if (CAUSAL) lim = min(lim, grow - kc0 + 1);
            if (lim < BN) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= lim) s[c] = -INFINITY;
            }
            const float mx = row_max_128(s);
            const float m_tile = mx * sl;
            float alpha = 1.f;
            if (m_tile > m + RESCALE_LOG2) {
                alpha = ex2(m - m_tile);
                m = m_tile;
            }
            const float base = (m == -INFINITY) ? 0.f : m;
            const uint64_t sl2 = f2_pack(sl, sl), nb2 = f2_pack(-base, -base);
            uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
            for (int c = 0; c < 2; ++c) {  // two halves of 64 keys
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(s[c * 64 + 2 * x], s[c * 64 + 2 * x + 1]), sl2, nb2), a0, a1);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    rs2[x & 1] = f2_add(rs2[x & 1], f2_pack(p0, p1));
                    hi[x] = pack_bf16x2(p0, p1);
                    if (NPROD == 3)
                        lo[x] = pack_bf16x2(p0 - __uint_as_float(hi[x] << 16), p1 - __uint_as_float(hi[x] & 0xFFFF0000u));
                }
                tmem_st32(tS + c * 32, hi);
                if (NPROD == 3) tmem_st32(tS + 64 + c * 32, lo);
            }
            float r0, r1;
            f2_unpack(f2_add(rs2[0], rs2[1]), r0, r1);
            l = l * alpha + (r0 + r1);
            if (NPROD == 1) {
                // as in the main kernel: the top weight's bf16 rounding joins O's normaliser
                const float p_top = ex2(fmaf(mx, sl, -base));
                dq = dq * alpha + (__uint_as_float(pack_bf16x2(p_top, 0.f) << 16) - p_top);
            }
            if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(tO + c * 32, raw);
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        float o0, o1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(raw[2 * x]), __uint_as_float(raw[2 * x + 1])), a2), o0, o1);
                        raw[2 * x] = __float_as_uint(o0);
                        raw[2 * x + 1] = __float_as_uint(o1);
                    }
                    tmem_st32(tO + c * 32, raw);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(&p_full));
        }
        if (ok && wait_or_abort(smem_addr(&o_full), 0, limit, &abort_flag)) {
            tc_fence_after();
            const float inv = prm.direct ? 1.f / (l + dq) : 1.f;
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
                uint32_t raw[32];
                tmem_ld32(tO + c * 32, raw);  // every lane loads; only rows < N store
                if (grow < N && prm.direct) {
                    const size_t e = ((size_t)bh * N + grow) * D + dv0 + c * 32;
                    if (prm.o_fp32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(prm.o) + e);
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            dst[x] = make_float4(__uint_as_float(raw[4 * x]) * inv, __uint_as_float(raw[4 * x + 1]) * inv,
                                                 __uint_as_float(raw[4 * x + 2]) * inv, __uint_as_float(raw[4 * x + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(prm.o) + e);
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(raw[8 * x + 0]) * inv, __uint_as_float(raw[8 * x + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * inv, __uint_as_float(raw[8 * x + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * inv, __uint_as_float(raw[8 * x + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * inv, __uint_as_float(raw[8 * x + 7]) * inv);
                            dst[x] = w;
                        }
                    }
                } else if (grow < N) {
                    float4 *dst = reinterpret_cast<float4 *>(prm.o_part + (part_row + grow) * D + dv0 + c * 32);
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        dst[x] = make_float4(__uint_as_float(raw[4 * x]), __uint_as_float(raw[4 * x + 1]),
                                             __uint_as_float(raw[4 * x + 2]), __uint_as_float(raw[4 * x + 3]));
                }
            }
            if (grow < N && dvc == 0) {
                if (prm.direct) {
                    if (prm.lse) prm.lse[(size_t)bh * N + grow] = (m + log2f(l)) * 0.69314718055994530942f;
                } else {
                    prm.m_part[part_row + grow] = m;
                    prm.l_part[part_row + grow] = l;
                    prm.d_part[part_row + grow] = dq;
                }
            }
        } else if (!abort_flag) {
            raise_wide(ERR_WAIT, &abort_flag);
        } else {
            atomicOr(&g_wide_error_word, ERR_WAIT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), for Q, K and V in one
// launch (blockIdx.y picks the tensor); four elements per thread.
struct SplitArgs {
    const float4 *x[3];
    uint2 *hi[3];
    uint2 *lo[3];
};

__global__ void fa_split_kernel(const SplitArgs a, size_t n4)
{
    const float4 *__restrict__ x = a.x[blockIdx.y];
    uint2 *__restrict__ hi = a.hi[blockIdx.y];
    uint2 *__restrict__ lo = a.lo[blockIdx.y];
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = x[i];
        const uint32_t h01 = pack_bf16x2(v.x, v.y), h23 = pack_bf16x2(v.z, v.w);
        const uint32_t l01 = pack_bf16x2(v.x - __uint_as_float(h01 << 16), v.y - __uint_as_float(h01 & 0xFFFF0000u));
        const uint32_t l23 = pack_bf16x2(v.z - __uint_as_float(h23 << 16), v.w - __uint_as_float(h23 & 0xFFFF0000u));
        hi[i] = make_uint2(h01, h23);
        lo[i] = make_uint2(l01, l23);
    }
}

// Merge of the per-split partial results, one CTA per query row and one
// float4 of the row per thread, every split's load in flight together.
template <typename Tout>
__global__ void __launch_bounds__(256)
fa_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ m_part,
                  const float *__restrict__ l_part, const float *__restrict__ d_part,
                  Tout *__restrict__ o, float *__restrict__ lse, int BH, int N, int D, int n_split)
{
    __shared__ float w_s[MAX_SPLITS];
    __shared__ float inv_s;
    const size_t row = blockIdx.x;
    const size_t stride = (size_t)BH * N;
    if (threadIdx.x < 32) {
        // warp 0: reference maximum, weights 2^(m_s - m), denominators
        const int s = threadIdx.x;
        const float ms = s < n_split ? m_part[s * stride + row] : -INFINITY;
        float M = ms;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float wt = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
        float L = wt != 0.f ? wt * l_part[s * stride + row] : 0.f;
        float Lq = wt != 0.f ? wt * (l_part[s * stride + row] + d_part[s * stride + row]) : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            L += __shfl_xor_sync(0xffffffffu, L, off);
            Lq += __shfl_xor_sync(0xffffffffu, Lq, off);
        }
        if (s < n_split) w_s[s] = wt;
        if (s == 0) {
            inv_s = 1.f / Lq;
            if (lse) lse[row] = (M + log2f(L)) * 0.69314718055994530942f;
        }
    }
    __syncthreads();
    const float inv = inv_s;
    for (int c = threadIdx.x * 4; c < D; c += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s = 0; s < n_split; ++s) {
            const float wt = w_s[s];
            if (wt == 0.f) continue;  // empty splits hold no partial O
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(o_part + (s * stride + row) * D + c));
            acc.x = fmaf(wt, v.x, acc.x);
            acc.y = fmaf(wt, v.y, acc.y);
            acc.z = fmaf(wt, v.z, acc.z);
            acc.w = fmaf(wt, v.w, acc.w);
        }
        Tout *dst = o + row * D + c;
        if constexpr (sizeof(Tout) == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
        }
    }
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

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// ------------------------------------------------------------------ planning
WidePlan wide_plan(const Problem &p, int max_splits)
{
    WidePlan w{};
    const bool fp32_in = p.in_dtype == 1;
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    w.ok = p.d % 128 == 0 && p.d <= 1024 && (fp32_in ? p.d >= 128 : p.d >= 256) && p.scale > 0.f &&
           p.B * p.H <= 65535 && plain_layout(p) && al16(p.q) && al16(p.k) && al16(p.v) && al16(p.o);
    if (!w.ok) return w;
    const int64_t BH = p.B * p.H;
    w.nprod = fp32_in ? 3 : 1;
    w.dv = (p.d % 256 == 0) ? 256 : 128;
    w.n_q = (int)((p.N + BM - 1) / BM);
    w.n_kv = (int)((p.N + BN - 1) / BN);
    w.n_dv = (int)(p.d / w.dv);
    const int64_t base = (int64_t)w.n_q * w.n_dv * BH;
    const int64_t target = (int64_t)sm_count();  // one wave: more splits only add partials to merge
    int splits = (int)std::min<int64_t>({(int64_t)std::max(1, std::min(max_splits, MAX_SPLITS)), (int64_t)w.n_kv,
                                         std::max<int64_t>(1, (target + base - 1) / base)});
    w.tiles_per_split = (w.n_kv + splits - 1) / splits;
    w.n_split = (w.n_kv + w.tiles_per_split - 1) / w.tiles_per_split;
    // workspace: bf16 hi/lo copies of fp32 inputs, then partials when split
    const size_t n = (size_t)(BH * p.N * p.d);
    size_t off = 0;
    if (fp32_in) {
        for (int i = 0; i < 6; ++i) { w.off_split[i] = off; off += align256(n * 2); }
    }
    if (w.n_split > 1) {
        w.off_opart = off; off += align256((size_t)w.n_split * n * 4);
        const size_t rows = (size_t)w.n_split * BH * p.N * 4;
        w.off_m = off; off += align256(rows);
        w.off_l = off; off += align256(rows);
        w.off_d = off; off += align256(rows);
    }
    w.workspace_bytes = off;
    return w;
}

cudaError_t launch_wide(const Problem &p, const WidePlan &w, void *workspace, cudaStream_t stream, uint32_t flags,
                        const char **detail)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t BH = p.B * p.H;
    const size_t n = (size_t)(BH * p.N * p.d);
    const void *qh = p.q, *kh = p.k, *vh = p.v, *ql = p.q, *kl = p.k, *vl = p.v;
    cudaError_t e;
    if (w.nprod == 3) {
        void *buf[6];
        for (int i = 0; i < 6; ++i) buf[i] = ws + w.off_split[i];
        SplitArgs sa;
        sa.x[0] = static_cast<const float4 *>(p.q);
        sa.x[1] = static_cast<const float4 *>(p.k);
        sa.x[2] = static_cast<const float4 *>(p.v);
        for (int t = 0; t < 3; ++t) {
            sa.hi[t] = static_cast<uint2 *>(buf[2 * t]);
            sa.lo[t] = static_cast<uint2 *>(buf[2 * t + 1]);
        }
        const size_t n4 = n / 4;
        const unsigned blocks = (unsigned)std::min<size_t>((n4 + 255) / 256, (size_t)sm_count() * 4);
        fa_split_kernel<<<dim3(blocks, 3), 256, 0, stream>>>(sa, n4);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        qh = buf[0]; ql = buf[1]; kh = buf[2]; kl = buf[3]; vh = buf[4]; vl = buf[5];
    }
    CUtensorMap m[6];
    const void *ptrs[6] = {qh, ql, kh, kl, vh, vl};
    for (int i = 0; i < 6; ++i)
        if (!make_map(&m[i], ptrs[i], BH, p.N, p.d)) {
            *detail = "cuTensorMapEncodeTiled failed or is unavailable";
            return cudaErrorInvalidValue;
        }
    WideParams prm{};
    prm.N = (int)p.N;
    prm.BH = (int)BH;
    prm.D = (int)p.d;
    prm.n_q = w.n_q;
    prm.n_dv = w.n_dv;
    prm.n_split = w.n_split;
    prm.tiles_per_split = w.tiles_per_split;
    prm.n_kv = w.n_kv;
    prm.scale_log2 = p.scale * 1.4426950408889634f;
    prm.wait_limit_ns = 2000000000ull;
    prm.direct = w.n_split == 1;
    prm.o = p.o;
    prm.o_fp32 = p.o_dtype == 1;
    prm.lse = p.lse;
    if (!prm.direct) {
        prm.o_part = reinterpret_cast<float *>(ws + w.off_opart);
        prm.m_part = reinterpret_cast<float *>(ws + w.off_m);
        prm.l_part = reinterpret_cast<float *>(ws + w.off_l);
        prm.d_part = reinterpret_cast<float *>(ws + w.off_d);
    }
    (void)flags;
    dim3 grid((unsigned)(w.n_q * w.n_dv * w.n_split), (unsigned)BH);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        kern<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5], prm);
        return cudaGetLastError();
    };
    if (w.nprod == 3) {
        if (w.dv == 256) e = p.causal ? go(fa_wide_kernel<3, 256, true>) : go(fa_wide_kernel<3, 256, false>);
        else e = p.causal ? go(fa_wide_kernel<3, 128, true>) : go(fa_wide_kernel<3, 128, false>);
    } else {
        if (w.dv == 256) e = p.causal ? go(fa_wide_kernel<1, 256, true>) : go(fa_wide_kernel<1, 256, false>);
        else e = p.causal ? go(fa_wide_kernel<1, 128, true>) : go(fa_wide_kernel<1, 128, false>);
    }
    if (e != cudaSuccess) return e;
    if (!prm.direct)
        e = launch_combine(prm.o_part, prm.m_part, prm.l_part, prm.d_part, p.o, p.o_dtype == 1, p.lse, BH, p.N,
                           (int)p.d, w.n_split, stream);
    return e;
}

cudaError_t launch_combine(const float *o_part, const float *m_part, const float *l_part, const float *d_part, void *o,
                           bool o_fp32, float *lse, int64_t BH, int64_t N, int D, int n_split, cudaStream_t stream)
{
    if (n_split < 1 || n_split > MAX_SPLITS || D % 4 != 0) return cudaErrorInvalidValue;
    const unsigned rows = (unsigned)(BH * N);
    const int threads = (int)std::min<int64_t>(256, std::max<int64_t>(32, D / 4));
    if (o_fp32)
        fa_combine_kernel<float><<<rows, threads, 0, stream>>>(o_part, m_part, l_part, d_part, static_cast<float *>(o),
                                                               lse, (int)BH, (int)N, D, n_split);
    else
        fa_combine_kernel<__nv_bfloat16><<<rows, threads, 0, stream>>>(
            o_part, m_part, l_part, d_part, static_cast<__nv_bfloat16 *>(o), lse, (int)BH, (int)N, D, n_split);
    return cudaGetLastError();
}

cudaError_t wide_error_word_ptr(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_wide_error_word);
}

}  // namespace fa
