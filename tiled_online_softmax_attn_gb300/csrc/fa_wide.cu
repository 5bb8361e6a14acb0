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

// ---------------------------------------------------------------------------
// Cluster form of the wide-head kernel, for head dimensions of 512 and 1024
// (R = d / 256 CTAs per cluster).  The R CTAs of a cluster share one query
// tile and one key range; CTA x owns the O slice of columns [256 x, 256 x +
// 256) and forms the partial scores S_x = Q[:, 256 x ...] K[:, 256 x ...]^T
// over its part of the head dimension, so S = sum_x S_x is formed once per
// cluster instead of once per O slice.  The partials meet in distributed
// shared memory, one 32-row quarter of the tile at a time:
//
//   * quarter w (tensor-memory lanes 32 w ...) is owned by CTA w % R.  Every
//     other CTA's warp w stages its 32 partial rows in its own shared memory
//     and one lane copies them (bulk copy engine) into the owner's receive
//     slot, completing the bytes on the owner's `recv_full`;
//   * the owner's warp w adds the R partials (its own first, then the others
//     in rank order), runs the online softmax of "Tiling the Loop" for the 32
//     rows (running maximum, weights, row sums; lazy rescaling as in the
//     single-CTA kernel), writes the weights (bf16 hi, and lo for fp32 inputs)
//     into its own tensor memory, and copies them, with each row's reference
//     maximum m and normaliser l + dq, into every other CTA's staging slot;
//   * each CTA's warp w takes the weights of its lanes from the staging slot
//     into tensor memory, rescales its O rows by alpha = 2^(m_old - m) (the
//     same instruction on the same values as the owner's), and the MMA warp
//     forms O_x += P V[:, 256 x ...] from there.
//
// No slot needs a "free" signal: a sender stages partial(j + 1) in its staging
// slot only after it has read the weights of tile j that arrived there, and
// the owner writes those only after every partial(j) has landed; the owner
// stages the copy of tile j for CTA y in y's own receive slot, which y
// refills with partial(j + 1) only after that copy has reached it.
//
// The CTAs of a cluster synchronise once after setup (nobody arrives on a
// barrier that is not initialised yet) and once before exit (nobody writes
// into the shared memory of a CTA that has left).  Every wait is bounded as
// in the rest of the library.
//
// Tensor memory: S partial [0, 128), P_hi [128, 192), P_lo [192, 256), O slice
// [256, 512).  Shared memory (all dynamic, 1024-byte aligned base checked at
// run time): a two-slot ring of 64 KB (the S chunks of the CTA's part of Q and
// K, then the V slice), the receive slots (32 rows x 128 fp32), the staging
// slots (32 rows x 128 bf16 hi + 128 lo) and 8-byte row records {m, l + dq},
// slots stored chunk-major (slot_chunk).  The epilogue stages the O slice in
// the ring, idle by then, and writes it row by row with the lanes of a warp on
// consecutive addresses.

template <int R>
struct ClLayout {
    static constexpr int OWNED = 4 / R;                  // row quarters a CTA owns
    static constexpr int FOREIGN = 4 - OWNED;            // quarters other CTAs own
    static constexpr uint32_t SLOT = 32 * 512;           // 32 rows x 512 bytes
    static constexpr uint32_t REC = 32 * 8;              // 32 row records {m, l + dq}
    static constexpr uint32_t OFF_RECV = 2 * STAGE_BYTES;                // [OWNED][R - 1] slots
    static constexpr uint32_t OFF_PST = OFF_RECV + OWNED * (R - 1) * SLOT;  // [FOREIGN] slots
    static constexpr uint32_t OFF_PREC = OFF_PST + FOREIGN * SLOT;         // [FOREIGN] incoming records
    static constexpr uint32_t OFF_OREC = OFF_PREC + FOREIGN * REC;         // [OWNED][R - 1] outgoing records
    static constexpr uint32_t OFF_BARS = OFF_OREC + OWNED * (R - 1) * REC;
    // barriers: full[2], empty[2], s_full, s_read, p_full, p_free, o_full, drain,
    // recv_full[2], pst_full[3]; then tensor-memory base and abort flag
    static constexpr uint32_t BAR_BYTES = 18 * 8 + 16;
    static constexpr uint32_t NEED = OFF_BARS + BAR_BYTES;
    static constexpr uint32_t SMEM_MAX = 232448;
    static constexpr uint32_t SMEM = NEED + 1024 <= SMEM_MAX ? NEED + 1024 : SMEM_MAX;
};
static_assert(ClLayout<4>::NEED <= ClLayout<4>::SMEM_MAX && ClLayout<2>::NEED <= ClLayout<2>::SMEM_MAX,
              "cluster kernel: shared memory above the 227 KB a CTA may use");

// Byte offset of 16-byte chunk c of row `row` in an exchange slot: chunk-major,
// so that the 32 lanes of a warp (one row each) touch 512 contiguous bytes.
__device__ __forceinline__ uint32_t slot_chunk(int row, int c) { return (uint32_t)(c * 512 + row * 16); }

constexpr uint32_t ERR_CL_LAYOUT = 256u;  // the cluster kernel's shared-memory layout did not fit its allocation

template <int NPROD, int R, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fa_wide_cluster_kernel(const __grid_constant__ CUtensorMap tm_qh, const __grid_constant__ CUtensorMap tm_ql,
                       const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_kl,
                       const __grid_constant__ CUtensorMap tm_vh, const __grid_constant__ CUtensorMap tm_vl,
                       const WideParams prm)
{
    using L = ClLayout<R>;
    constexpr int DVC = 256;                       // O columns per CTA
    constexpr uint32_t P_BYTES = NPROD == 3 ? L::SLOT : L::SLOT / 2;  // chunk-major: hi chunks first
    extern __shared__ uint8_t smem_raw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, D = prm.D;
    const int x = (int)(blockIdx.x % R);           // rank in the cluster = O slice = part of d
    const int cl = (int)(blockIdx.x / R);
    const int qt = CAUSAL ? prm.n_q - 1 - cl / prm.n_split : cl / prm.n_split;
    const int sp = cl % prm.n_split;
    const int bh = (int)blockIdx.y;
    const int q0 = qt * BM, dv0 = x * DVC, dk0 = x * DVC;
    const int kv_need = CAUSAL ? min(prm.n_kv, qt + 1) : prm.n_kv;
    const int kv_lo = sp * prm.tiles_per_split;
    const int n_j = min(kv_lo + prm.tiles_per_split, kv_need) - kv_lo;
    const size_t part_row = ((size_t)sp * prm.BH + bh) * N;

    if (n_j <= 0) {  // every CTA of the cluster takes this branch: an empty partial
        if (!prm.direct && x == 0 && warp < 4) {
            const int grow = q0 + (int)threadIdx.x;
            if (grow < N) {
                prm.m_part[part_row + grow] = -INFINITY;
                prm.l_part[part_row + grow] = 0.f;
                prm.d_part[part_row + grow] = 0.f;
            }
        }
        return;
    }
    // 1024-byte aligned base (every CTA of the cluster gets the same offset, so
    // all of them leave here together if the layout does not fit)
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    if (pad + L::NEED > L::SMEM) {
        if (threadIdx.x == 0) atomicOr(&g_wide_error_word, ERR_CL_LAYOUT);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    const uint32_t s_base = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BARS);
    uint64_t *full_b = bars, *empty_b = bars + 2;
    uint64_t &s_full = bars[4], &s_read = bars[5], &p_full = bars[6], &p_free = bars[7], &o_full = bars[8],
             &drain = bars[9];
    uint64_t *recv_full = bars + 10, *pst_full = bars + 12;
    uint32_t &tmem_base_s = *reinterpret_cast<uint32_t *>(smem + L::OFF_BARS + 18 * 8);
    volatile int &abort_flag = *reinterpret_cast<volatile int *>(smem + L::OFF_BARS + 18 * 8 + 4);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty_b[s]), 1);
        }
        mbar_init(smem_addr(&s_full), 1);
        mbar_init(smem_addr(&s_read), 128);
        mbar_init(smem_addr(&p_full), 128);
        mbar_init(smem_addr(&p_free), 1);
        mbar_init(smem_addr(&o_full), 1);
        mbar_init(smem_addr(&drain), 1);
        for (int i = 0; i < 2; ++i) mbar_init(smem_addr(&recv_full[i]), 1);  // the owner's expect_tx
        for (int i = 0; i < 3; ++i) mbar_init(smem_addr(&pst_full[i]), 1);   // the receiver's expect_tx
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(&tmem_base_s), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peers' barriers are initialised before anyone arrives on them
    tc_fence_after();
    pdl_launch_dependents();  // the merge kernel may be scheduled; it waits for this one
    pdl_wait_prior();         // the split pass's bf16 copies are complete and visible
    const uint32_t tmem = tmem_base_s;
    const uint64_t limit = prm.wait_limit_ns;

    if (warp == TMA_WARP) {
        // ================================================================ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int it = 0;
            bool ok = true;
            auto acquire = [&](uint32_t bytes) -> int {
                const int st = it & 1;
                if (!wait_or_abort(smem_addr(&empty_b[st]), (uint32_t)(((it >> 1) & 1) ^ 1), limit, &abort_flag))
                    return -1;
                mbar_arrive_expect_tx(smem_addr(&full_b[st]), bytes);
                return st;
            };
            auto load_s = [&](int jj) {
                const int k0 = (kv_lo + jj) * BN;
                for (int c = 0; ok && c < DVC / 64; ++c) {
                    const int st = acquire(NPROD == 3 ? 4 * BOX_BYTES : 2 * BOX_BYTES);
                    if (st < 0) { ok = false; break; }
                    const uint32_t dst = s_base + st * STAGE_BYTES, fb = smem_addr(&full_b[st]);
                    tma_load_3d(dst, &tm_qh, fb, dk0 + c * 64, q0, bh, pol);
                    tma_load_3d(dst + 2 * BOX_BYTES, &tm_kh, fb, dk0 + c * 64, k0, bh, pol);
                    if (NPROD == 3) {
                        tma_load_3d(dst + BOX_BYTES, &tm_ql, fb, dk0 + c * 64, q0, bh, pol);
                        tma_load_3d(dst + 3 * BOX_BYTES, &tm_kl, fb, dk0 + c * 64, k0, bh, pol);
                    }
                    ++it;
                }
            };
            auto load_v = [&](int jj) {
                const int k0 = (kv_lo + jj) * BN;
                for (int part = 0; ok && part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = acquire((DVC / 64) * BOX_BYTES);
                    if (st < 0) { ok = false; break; }
                    const uint32_t dst = s_base + st * STAGE_BYTES, fb = smem_addr(&full_b[st]);
                    for (int a = 0; a < DVC / 64; ++a)
                        tma_load_3d(dst + a * BOX_BYTES, part ? &tm_vl : &tm_vh, fb, dv0 + a * 64, k0, bh, pol);
                    ++it;
                }
            };
            // the order the MMA warp consumes: S(0), then S(j), V(j - 1) ..., then V(last)
            for (int jj = 0; ok && jj < n_j; ++jj) {
                load_s(jj);
                if (jj > 0) load_v(jj - 1);
            }
            if (ok) load_v(n_j - 1);
            if (!ok) {
                if (!abort_flag) raise_wide(ERR_WAIT, &abort_flag);
                for (int j = max(0, it - 2); j < it; ++j)
                    if (!mbar_wait_bounded(smem_addr(&full_b[j & 1]), (uint32_t)((j >> 1) & 1), limit))
                        atomicOr(&g_wide_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================================================================ MMA issuer
        {
            const uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(BM, DVC, 0, 1);
            const uint32_t tS = tmem, tPh = tmem + 128, tPl = tmem + 192, tO = tmem + COL_O;
            int it = 0;
            bool ok = true, issued = false;
            auto wait_full = [&]() -> int {
                const int st = it & 1;
                if (!wait_or_abort_w(smem_addr(&full_b[st]), (uint32_t)((it >> 1) & 1), limit, &abort_flag))
                    return -1;
                tc_fence_after();
                return st;
            };
            auto mma_s = [&](int jj) -> bool {
                if (jj > 0 && !wait_or_abort_w(smem_addr(&s_read), (uint32_t)((jj - 1) & 1), limit, &abort_flag))
                    return false;
                tc_fence_after();
                for (int c = 0; c < DVC / 64; ++c) {
                    const int st = wait_full();
                    if (st < 0) return false;
                    const uint32_t base = s_base + st * STAGE_BYTES;
                    const uint64_t dqh = sdesc_sw128(base, 16, 1024), dql = sdesc_sw128(base + BOX_BYTES, 16, 1024);
                    const uint64_t dkh = sdesc_sw128(base + 2 * BOX_BYTES, 16, 1024),
                                   dkl = sdesc_sw128(base + 3 * BOX_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t off = (uint64_t)(kk * 2);
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
                mma_commit_w(smem_addr(&s_full));
                return true;
            };
            auto mma_pv = [&](int jj) -> bool {
                if (!wait_or_abort_w(smem_addr(&p_full), (uint32_t)(jj & 1), limit, &abort_flag)) return false;
                tc_fence_after();
                for (int part = 0; part < (NPROD == 3 ? 2 : 1); ++part) {
                    const int st = wait_full();
                    if (st < 0) return false;
                    const uint64_t dv = sdesc_sw128(s_base + st * STAGE_BYTES, BOX_BYTES, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t voff = (uint64_t)((kk * 16 * 128) >> 4);
                        if (part == 0) {
                            mma_ts_w(tO, tPh + kk * 8, dv + voff, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                            if (NPROD == 3) mma_ts_w(tO, tPl + kk * 8, dv + voff, idesc_o, 1u);
                        } else {
                            mma_ts_w(tO, tPh + kk * 8, dv + voff, idesc_o, 1u);
                        }
                    }
                    issued = true;
                    mma_commit_w(smem_addr(&empty_b[st]));
                    ++it;
                }
                mma_commit_w(smem_addr(&p_free));
                return true;
            };
            for (int jj = 0; ok && jj < n_j; ++jj) {
                if (!mma_s(jj)) { ok = false; break; }
                if (jj > 0 && !mma_pv(jj - 1)) { ok = false; break; }
            }
            if (ok && !mma_pv(n_j - 1)) ok = false;
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
        // ================================================================ score exchange, softmax, epilogue
        const int w = warp;                          // row quarter: tensor-memory lanes 32 w ...
        const int r = w * 32 + lane;
        const int grow = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
        const uint32_t tS = lane_base, tPh = lane_base + 128, tPl = lane_base + 192, tO = lane_base + COL_O;
        const float sl = prm.scale_log2;
        const int owner = w % R;
        const bool is_owner = owner == x;
        const int oi = w / R;                        // index of quarter w among its owner's quarters
        // index of quarter w among CTA y's foreign quarters (w not owned by y)
        auto foreign_index = [](int y, int ww) { int f = 0; for (int v = 0; v < ww; ++v) f += (v % R != y); return f; };
        auto other_index = [](int y, int o) { return y < o ? y : y - 1; };  // rank y among the CTAs other than o
        float m = -INFINITY, l = 0.f, dq = 0.f;     // owner: running statistics; others: m and l + dq
        bool ok = true;
        auto fail = [&]() {
            ok = false;
            if (!abort_flag) raise_wide(ERR_WAIT, &abort_flag);
            else atomicOr(&g_wide_error_word, ERR_WAIT);
        };
        // Bounded waits with one outcome for the whole warp, so that the
        // warp-collective tensor-memory accesses after them stay converged.
        auto uwait = [&](const uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(smem_addr(bar), parity, limit, &abort_flag));
        };
        auto uwait_cl = [&](const uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort_cluster(smem_addr(bar), parity, limit, &abort_flag));
        };
        const int fi = is_owner ? 0 : foreign_index(x, w);
        for (int jj = 0; ok && jj < n_j; ++jj) {
            if (!uwait(&s_full, (uint32_t)(jj & 1))) { fail(); break; }
            tc_fence_after();
            float s[BN];
            {
                uint32_t raw[BN];
                tmem_ld128(tS, raw);
#pragma unroll
                for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(raw[c]);
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&s_read));          // the next S partial may overwrite tensor memory
            uint32_t ph[64], pl[64];                  // this row's weights, bf16 pairs
            float alpha = 1.f;
            if (is_owner) {
                // ---- sum the partials of the other CTAs into this row
                if (lane == 0)
                    mbar_arrive_expect_tx(smem_addr(&recv_full[oi]), (uint32_t)(R - 1) * L::SLOT);
                if (!uwait_cl(&recv_full[oi], (uint32_t)(jj & 1))) { fail(); break; }
                for (int y = 0; y < R; ++y) {
                    if (y == x) continue;
                    const uint8_t *slot = smem + L::OFF_RECV + (oi * (R - 1) + other_index(y, x)) * L::SLOT;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float4 v = *reinterpret_cast<const float4 *>(slot + slot_chunk(lane, c));
                        s[4 * c] += v.x;
                        s[4 * c + 1] += v.y;
                        s[4 * c + 2] += v.z;
                        s[4 * c + 3] += v.w;
                    }
                }
                // ---- online softmax of the row
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
                if (m_tile > m + RESCALE_LOG2) {
                    alpha = ex2(m - m_tile);
                    m = m_tile;
                }
                const float base = (m == -INFINITY) ? 0.f : m;
                const uint64_t sl2 = f2_pack(sl, sl), nb2 = f2_pack(-base, -base);
                uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl2, nb2), a0, a1);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    rs2[c & 1] = f2_add(rs2[c & 1], f2_pack(p0, p1));
                    ph[c] = pack_bf16x2(p0, p1);
                    pl[c] = NPROD == 3 ? pack_bf16x2(p0 - __uint_as_float(ph[c] << 16),
                                                     p1 - __uint_as_float(ph[c] & 0xFFFF0000u))
                                       : 0u;
                }
                float r0, r1;
                f2_unpack(f2_add(rs2[0], rs2[1]), r0, r1);
                l = l * alpha + (r0 + r1);
                if (NPROD == 1) {
                    const float p_top = ex2(fmaf(mx, sl, -base));
                    dq = dq * alpha + (__uint_as_float(pack_bf16x2(p_top, 0.f) << 16) - p_top);
                }
                // ---- the weights and {m, l + dq} to every other CTA: staged in that
                // CTA's own receive slot (its partial has been read), one bulk copy each
                for (int y = 0; y < R; ++y) {
                    if (y == x) continue;
                    const int k = oi * (R - 1) + other_index(y, x);
                    uint8_t *stg = smem + L::OFF_RECV + k * L::SLOT;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        *reinterpret_cast<uint4 *>(stg + slot_chunk(lane, c)) =
                            make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
                    if (NPROD == 3) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            *reinterpret_cast<uint4 *>(stg + slot_chunk(lane, 16 + c)) =
                                make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
                    }
                    *reinterpret_cast<float2 *>(smem + L::OFF_OREC + k * L::REC + lane * 8) = make_float2(m, l + dq);
                }
                fence_proxy_async_smem();            // the staged bytes are visible to the bulk copies
                __syncwarp();
                if (lane == 0) {
                    for (int y = 0; y < R; ++y) {
                        if (y == x) continue;
                        const int k = oi * (R - 1) + other_index(y, x);
                        const int fy = foreign_index(y, w);
                        const uint32_t bar = mapa_shared(smem_addr(&pst_full[fy]), (uint32_t)y);
                        bulk_copy_s2cluster(mapa_shared(s_base + L::OFF_PST + fy * L::SLOT, (uint32_t)y),
                                            s_base + L::OFF_RECV + k * L::SLOT, P_BYTES, bar);
                        bulk_copy_s2cluster(mapa_shared(s_base + L::OFF_PREC + fy * L::REC, (uint32_t)y),
                                            s_base + L::OFF_OREC + k * L::REC, L::REC, bar);
                    }
                }
            } else {
                // ---- send this row's partial to the owner, take the weights back
                uint8_t *stg = smem + L::OFF_PST + fi * L::SLOT;  // free: its last weights were read
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    *reinterpret_cast<float4 *>(stg + slot_chunk(lane, c)) =
                        make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // arm the slot for the weights of this tile before they can arrive
                    mbar_arrive_expect_tx(smem_addr(&pst_full[fi]), P_BYTES + L::REC);
                    const int k = oi * (R - 1) + other_index(x, owner);
                    bulk_copy_s2cluster(mapa_shared(s_base + L::OFF_RECV + k * L::SLOT, (uint32_t)owner),
                                        s_base + L::OFF_PST + fi * L::SLOT, L::SLOT,
                                        mapa_shared(smem_addr(&recv_full[oi]), (uint32_t)owner));
                }
                if (!uwait_cl(&pst_full[fi], (uint32_t)(jj & 1))) { fail(); break; }
                const uint8_t *pslot = smem + L::OFF_PST + fi * L::SLOT;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(pslot + slot_chunk(lane, c));
                    ph[4 * c] = v.x;
                    ph[4 * c + 1] = v.y;
                    ph[4 * c + 2] = v.z;
                    ph[4 * c + 3] = v.w;
                }
                if (NPROD == 3) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(pslot + slot_chunk(lane, 16 + c));
                        pl[4 * c] = v.x;
                        pl[4 * c + 1] = v.y;
                        pl[4 * c + 2] = v.z;
                        pl[4 * c + 3] = v.w;
                    }
                }
                const float2 rec = *reinterpret_cast<const float2 *>(smem + L::OFF_PREC + fi * L::REC + lane * 8);
                if (rec.x != m) alpha = ex2(m - rec.x);  // the owner's alpha: same instruction, same inputs
                m = rec.x;
                l = rec.y;                            // l + dq
            }
            // ---- this CTA's copy of the weights; O rows rescaled once the previous P V is done
            if (jj > 0 && !uwait(&p_free, (uint32_t)((jj - 1) & 1))) { fail(); break; }
            tc_fence_after();
            if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < DVC / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(tO + c * 32, raw);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float o0, o1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(raw[2 * e]), __uint_as_float(raw[2 * e + 1])), a2), o0, o1);
                        raw[2 * e] = __float_as_uint(o0);
                        raw[2 * e + 1] = __float_as_uint(o1);
                    }
                    tmem_st32(tO + c * 32, raw);
                }
            }
            {
                uint32_t h32[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) h32[c] = ph[c];
                tmem_st32(tPh, h32);
#pragma unroll
                for (int c = 0; c < 32; ++c) h32[c] = ph[32 + c];
                tmem_st32(tPh + 32, h32);
                if (NPROD == 3) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) h32[c] = pl[c];
                    tmem_st32(tPl, h32);
#pragma unroll
                    for (int c = 0; c < 32; ++c) h32[c] = pl[32 + c];
                    tmem_st32(tPl + 32, h32);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_addr(&p_full));
        }
        if (ok && uwait(&o_full, 0)) {
            tc_fence_after();
            // O rows through shared memory: thread r writes its row (256 fp32,
            // chunks rotated by the row so the warp's stores spread over the
            // banks), then the warp writes each of its 32 rows with its lanes on
            // consecutive addresses.  Warp w uses its own 32 KB of the ring.
            const float inv = prm.direct ? 1.f / (is_owner ? l + dq : l) : 1.f;
            uint8_t *stage = smem + (uint32_t)w * 32 * (DVC * 4);
            fence_proxy_async_smem();
#pragma unroll 1
            for (int c = 0; c < DVC / 32; ++c) {
                uint32_t raw[32];
                tmem_ld32(tO + c * 32, raw);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int ch = c * 8 + q;  // float4 chunk of the row, 0..63
                    *reinterpret_cast<float4 *>(stage + lane * (DVC * 4) + (((ch ^ lane) & 63) << 4)) =
                        make_float4(__uint_as_float(raw[4 * q]) * inv, __uint_as_float(raw[4 * q + 1]) * inv,
                                    __uint_as_float(raw[4 * q + 2]) * inv, __uint_as_float(raw[4 * q + 3]) * inv);
                }
            }
            __syncwarp();
            for (int rr = 0; rr < 32; ++rr) {
                const int g = q0 + w * 32 + rr;
                if (g >= N) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = h * 32 + lane;
                    const float4 v = *reinterpret_cast<const float4 *>(stage + rr * (DVC * 4) + (((ch ^ rr) & 63) << 4));
                    if (!prm.direct) {
                        reinterpret_cast<float4 *>(prm.o_part + (part_row + g) * D + dv0)[ch] = v;
                    } else if (prm.o_fp32) {
                        reinterpret_cast<float4 *>(static_cast<float *>(prm.o) + ((size_t)bh * N + g) * D + dv0)[ch] = v;
                    } else {
                        reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(prm.o) + ((size_t)bh * N + g) * D + dv0)[ch] =
                            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                    }
                }
            }
            if (grow < N && is_owner) {  // the row statistics, from the CTA that computed them
                if (prm.direct) {
                    if (prm.lse) prm.lse[(size_t)bh * N + grow] = (m + log2f(l)) * 0.69314718055994530942f;
                } else {
                    prm.m_part[part_row + grow] = m;
                    prm.l_part[part_row + grow] = l;
                    prm.d_part[part_row + grow] = dq;
                }
            }
        } else if (ok) {
            if (!abort_flag) raise_wide(ERR_WAIT, &abort_flag);
            else atomicOr(&g_wide_error_word, ERR_WAIT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (abort_flag) {
        // After a wait gave up, a peer's bulk copy toward this CTA may still be
        // in flight (nobody waits for it any more): give it time to land before
        // the shared memory is released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000ull) {
        }
    }
    cluster_sync_all();  // no peer writes into this CTA's shared memory after it exits
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), for Q, K and V in one
// launch (blockIdx.y picks the tensor).  A block converts SPLIT_PER_BLOCK
// float4 groups, four per thread, all four loads issued before any store (the
// fp32 inputs are read once: streaming loads).
struct SplitArgs {
    const float4 *x[4];
    uint2 *hi[4];
    uint2 *lo[4];
};
constexpr int SPLIT_THREADS = 256, SPLIT_UNROLL = 4, SPLIT_PER_BLOCK = SPLIT_THREADS * SPLIT_UNROLL;

__global__ void __launch_bounds__(SPLIT_THREADS) fa_split_kernel(const __grid_constant__ SplitArgs a, size_t n4)
{
    const float4 *__restrict__ x = a.x[blockIdx.y];
    uint2 *__restrict__ hi = a.hi[blockIdx.y];
    uint2 *__restrict__ lo = a.lo[blockIdx.y];
    const size_t i0 = (size_t)blockIdx.x * SPLIT_PER_BLOCK + threadIdx.x;
    float4 v[SPLIT_UNROLL];
#pragma unroll
    for (int u = 0; u < SPLIT_UNROLL; ++u) {
        const size_t i = i0 + (size_t)u * SPLIT_THREADS;
        if (i < n4) v[u] = __ldcs(x + i);
    }
    pdl_launch_dependents();  // the attention kernel's prologue may overlap the stores
#pragma unroll
    for (int u = 0; u < SPLIT_UNROLL; ++u) {
        const size_t i = i0 + (size_t)u * SPLIT_THREADS;
        if (i >= n4) break;
        const uint32_t h01 = pack_bf16x2(v[u].x, v[u].y), h23 = pack_bf16x2(v[u].z, v[u].w);
        const uint32_t l01 = pack_bf16x2(v[u].x - __uint_as_float(h01 << 16), v[u].y - __uint_as_float(h01 & 0xFFFF0000u));
        const uint32_t l23 = pack_bf16x2(v[u].z - __uint_as_float(h23 << 16), v[u].w - __uint_as_float(h23 & 0xFFFF0000u));
        hi[i] = make_uint2(h01, h23);
        lo[i] = make_uint2(l01, l23);
    }
}

// Merge of the per-split partial results ("Core FlashAttention Mechanics",
// item 3: rescale each partial by 2^(m_s - M) and divide by the rescaled sum).
// COMBINE_COLS columns of a row per thread, D / COMBINE_COLS threads per row,
// as many rows as fit in 256 threads per block (two blocks per SM: one wave
// for the d = 1024 rows of a 1024-row head).  Every thread loads the maxima,
// sums and partial rows of the first HOLD splits itself (one round trip to
// memory, no block barrier); further splits are loaded as they are used.
constexpr int COMBINE_THREADS = 256, COMBINE_COLS = 16;

template <typename Tout>
__global__ void __launch_bounds__(COMBINE_THREADS, 2)
fa_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ m_part,
                  const float *__restrict__ l_part, const float *__restrict__ d_part,
                  Tout *__restrict__ o, float *__restrict__ lse, int BH, int N, int D, int n_split)
{
    constexpr int V = COMBINE_COLS / 4;  // float4 per thread and split
    const int tpr = D / COMBINE_COLS, per_block = COMBINE_THREADS / tpr;  // threads per row, rows per block
    const size_t rows = (size_t)BH * N;
    const int r = (int)threadIdx.x / tpr;
    const size_t row = (size_t)blockIdx.x * per_block + r;
    const int c0 = (int)(threadIdx.x % tpr) * COMBINE_COLS;
    pdl_wait_prior();  // the partials come from the kernel before this one
    if (r >= per_block || row >= rows) return;
    constexpr int HOLD = 4;
    const size_t ostep = rows * (size_t)D;  // elements between two splits' partial O
    const float *op = o_part + row * D + c0, *mp = m_part + row, *lp = l_part + row, *dp = d_part + row;
    float4 x[HOLD][V];
    float ms[HOLD], ls[HOLD], ds[HOLD];
#pragma unroll
    for (int s = 0; s < HOLD; ++s) {
        ms[s] = -INFINITY;
        if (s < n_split) {
#pragma unroll
            for (int v = 0; v < V; ++v) x[s][v] = __ldcs(reinterpret_cast<const float4 *>(op + s * ostep) + v);
            ms[s] = mp[s * rows];
            ls[s] = lp[s * rows];
            ds[s] = dp[s * rows];
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < HOLD; ++s) M = fmaxf(M, ms[s]);
#pragma unroll 1
    for (int s = HOLD; s < n_split; ++s) M = fmaxf(M, mp[s * rows]);
    float L = 0.f, Lq = 0.f;
    float4 acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float m_s, float l_s, float d_s, const float4 (&y)[V]) {
        if (m_s == -INFINITY) return;  // an empty split holds no partial O
        const float wt = exp2f(m_s - M);
        L = fmaf(wt, l_s, L);
        Lq = fmaf(wt, l_s + d_s, Lq);
#pragma unroll
        for (int v = 0; v < V; ++v)
            acc[v] = make_float4(fmaf(wt, y[v].x, acc[v].x), fmaf(wt, y[v].y, acc[v].y), fmaf(wt, y[v].z, acc[v].z),
                                 fmaf(wt, y[v].w, acc[v].w));
    };
#pragma unroll
    for (int s = 0; s < HOLD; ++s)
        if (s < n_split) add(ms[s], ls[s], ds[s], x[s]);
#pragma unroll 1
    for (int s = HOLD; s < n_split; ++s) {
        float4 y[V];
#pragma unroll
        for (int v = 0; v < V; ++v) y[v] = __ldcs(reinterpret_cast<const float4 *>(op + s * ostep) + v);
        add(mp[s * rows], lp[s * rows], dp[s * rows], y);
    }
    const float inv = 1.f / Lq;
    Tout *dst = o + row * D + c0;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float4 a = acc[v];
        if constexpr (sizeof(Tout) == 4)
            reinterpret_cast<float4 *>(dst)[v] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        else
            reinterpret_cast<uint2 *>(dst)[v] = make_uint2(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv));
    }
    if (lse && c0 == 0) lse[row] = (M + log2f(L)) * 0.69314718055994530942f;
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
    // d = 512 and 1024: the CTAs of one query tile form S once as a cluster
    w.cluster = (p.d == 512 || p.d == 1024) ? (int)(p.d / 256) : 1;
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
        const unsigned blocks = (unsigned)((n4 + SPLIT_PER_BLOCK - 1) / SPLIT_PER_BLOCK);
        fa_split_kernel<<<dim3(blocks, 3), SPLIT_THREADS, 0, stream>>>(sa, n4);
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
    if (w.cluster > 1) {
        // grid.x = (query tile, split) clusters of R CTAs, one O slice each
        bool no_room = false;  // set when the GPU cannot hold even one cluster of this size
        auto go_cl = [&](auto kern, int smem) -> cudaError_t {
            cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (err != cudaSuccess) return err;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(NUM_THREADS, 1, 1);
            cfg.dynamicSmemBytes = (size_t)smem;
            cfg.stream = stream;
            cudaLaunchAttribute at[2];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)w.cluster;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            // the prologue may overlap the split pass's tail (the kernel waits for it
            // before its first global access)
            at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            at[1].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = at;
            cfg.numAttrs = w.nprod == 3 ? 2 : 1;
            // a GPU partition may have too few SMs per cluster slot: asked once per
            // device and cluster size
            static int fits[64][5];  // 0 unknown, 1 fits, 2 does not
            int dev = 0;
            if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
            int &f = fits[dev & 63][w.cluster];
            if (f == 0) {
                int n = 0;
                cudaLaunchConfig_t one = cfg;
                one.numAttrs = 1;
                f = (cudaOccupancyMaxActiveClusters(&n, kern, &one) == cudaSuccess && n > 0) ? 1 : 2;
                (void)cudaGetLastError();
            }
            if (f == 2) {
                no_room = true;
                return cudaSuccess;
            }
            return cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], m[5], prm);
        };
        constexpr int S4 = (int)ClLayout<4>::SMEM, S2 = (int)ClLayout<2>::SMEM;
        if (w.nprod == 3) {
            if (w.cluster == 4) e = p.causal ? go_cl(fa_wide_cluster_kernel<3, 4, true>, S4) : go_cl(fa_wide_cluster_kernel<3, 4, false>, S4);
            else e = p.causal ? go_cl(fa_wide_cluster_kernel<3, 2, true>, S2) : go_cl(fa_wide_cluster_kernel<3, 2, false>, S2);
        } else {
            if (w.cluster == 4) e = p.causal ? go_cl(fa_wide_cluster_kernel<1, 4, true>, S4) : go_cl(fa_wide_cluster_kernel<1, 4, false>, S4);
            else e = p.causal ? go_cl(fa_wide_cluster_kernel<1, 2, true>, S2) : go_cl(fa_wide_cluster_kernel<1, 2, false>, S2);
        }
        if (no_room) {
            // no room for a cluster of this size: the single-CTA kernel below
            // computes the same result
        } else {
            if (e != cudaSuccess) return e;
            if (!prm.direct)
                e = launch_combine(prm.o_part, prm.m_part, prm.l_part, prm.d_part, p.o, p.o_dtype == 1, p.lse, BH, p.N,
                                   (int)p.d, w.n_split, stream);
            return e;
        }
    }
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

cudaError_t launch_split_hilo(const float *const *x, void *const *hi, void *const *lo, int count, size_t n,
                              cudaStream_t stream)
{
    if (count < 1 || count > 4 || n % 4 != 0) return cudaErrorInvalidValue;
    SplitArgs sa{};
    for (int t = 0; t < count; ++t) {
        sa.x[t] = reinterpret_cast<const float4 *>(x[t]);
        sa.hi[t] = static_cast<uint2 *>(hi[t]);
        sa.lo[t] = static_cast<uint2 *>(lo[t]);
    }
    const size_t n4 = n / 4;
    const unsigned blocks = (unsigned)((n4 + SPLIT_PER_BLOCK - 1) / SPLIT_PER_BLOCK);
    fa_split_kernel<<<dim3(blocks, (unsigned)count), SPLIT_THREADS, 0, stream>>>(sa, n4);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *o_part, const float *m_part, const float *l_part, const float *d_part, void *o,
                           bool o_fp32, float *lse, int64_t BH, int64_t N, int D, int n_split, cudaStream_t stream)
{
    if (n_split < 1 || n_split > MAX_SPLITS || D % COMBINE_COLS != 0 || D > COMBINE_COLS * COMBINE_THREADS)
        return cudaErrorInvalidValue;
    const int64_t per_block = COMBINE_THREADS / (D / COMBINE_COLS);
    const unsigned blocks = (unsigned)((BH * N + per_block - 1) / per_block);
    // programmatic dependent launch: the merge's blocks may be scheduled while
    // the attention kernel finishes; they wait for it before reading (pdl_wait_prior)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(COMBINE_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (o_fp32)
        return cudaLaunchKernelEx(&cfg, fa_combine_kernel<float>, o_part, m_part, l_part, d_part, static_cast<float *>(o),
                                  lse, (int)BH, (int)N, D, n_split);
    return cudaLaunchKernelEx(&cfg, fa_combine_kernel<__nv_bfloat16>, o_part, m_part, l_part, d_part,
                              static_cast<__nv_bfloat16 *>(o), lse, (int)BH, (int)N, D, n_split);
}

cudaError_t wide_error_word_ptr(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_wide_error_word);
}

}  // namespace fa
