// Tensor-core backward pass (tcgen05 + TMA), bf16 inputs, d in {64, 128}.
//
// The gradients of the forward pass by recomputation from the stored per-row
// log-sum-exp ("FlashAttention", ai360xpert.com, "Recomputation in the
// backward pass"); definitions as in fa_backward.cu.  Two kernels, neither of
// which accumulates across CTAs:
//
//   dK/dV kernel -- a CTA owns 128 keys (one per tensor-memory lane) and
//   streams the query tiles that see them.  Per query tile:
//     S^T  = K_j Q_i^T       (SS MMA)          -> TMEM
//     dP^T = V_j dO_i^T      (SS MMA)          -> TMEM
//     P^T  = exp2(S^T scale log2 e - LSE_i log2 e)   (elementwise warps)
//     dV  += P^T dO_i        (A = P^T from TMEM, B = dO_i MN-major)
//     dS^T = P^T (dP^T - delta_i)
//     dK  += dS^T Q_i        (A = dS^T from TMEM, B = Q_i MN-major)
//   P^T and dS^T are written as bf16 over the dP^T columns once those are in
//   registers, so S^T(i+1) is computed while the warps work on tile i.
//   dQ kernel -- a CTA owns 128 queries and streams the key tiles they see:
//     S = Q_i K_j^T, dP = dO_i V_j^T, dS = P (dP - delta), dQ += dS K_j.
//
// So S and dP are formed twice (7 products of 128 x 128 x d instead of 5):
// the price of no atomics and deterministic gradients.  Eight elementwise
// warps do the elementwise work: warp w reads tensor-memory lanes
// 32 (w % 4) .. + 31 (one row per thread) and the half w / 4 of the 128
// columns, so two warps share each row and each SM sub-partition runs two of
// them; no reduction crosses columns.  Warp 8 issues the TMA loads, warp 9 the
// MMAs.  The two score products of a tile signal separate barriers, so the
// exponentials start as soon as the first is done.  The two streamed tiles
// travel in rings of their own (full/empty barrier pair per slot), so the one
// read first lands first and its ring can be the deeper one.
// Every wait is bounded as in the forward kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace fa {

__device__ uint32_t g_bwd_error_word;

namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = 128;
// Elementwise warps: 4 lane quarters x NH column groups of W = 128 / NH columns.
// Two groups for both head dimensions: four groups at d = 64 (16 elementwise
// warps) measured no faster, the d = 64 step being bound by the issue of its
// 24 MMAs (16 of them N = 64) rather than by the elementwise work.
__host__ __device__ constexpr int ew_groups(int) { return 2; }
template <int D>
struct EW {
    static constexpr int NH = ew_groups(D);
    static constexpr int W = BM / NH;               // columns per elementwise thread
    static constexpr int WARPS = 4 * NH;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int NUM_THREADS = THREADS + 64;
    static constexpr int TMA_WARP = WARPS;
    static constexpr int MMA_WARP = WARPS + 1;
};
constexpr uint32_t TMEM_COLS = 512;
constexpr int PERSIST_MAX_COLS = 2048;  // persistent CTAs for items of at most this many tiles x d
constexpr uint32_t BOX = 128 * 128;  // one 128-row x 64-column bf16 box
constexpr uint32_t VEC_BYTES = 1024;  // lse2 and delta of 128 rows

// Barriers and flags of the dK/dV kernel, kept at the end of its dynamic shared
// memory: at d = 128 its tiles take all but a few hundred bytes of the 227 KB a
// CTA may have, so nothing is left for static shared memory.
struct KvBars {
    uint64_t res_full, res_empty, st_full, s_read, dp_full, p_ready, ds_ready, o_full, acc_empty, drain;
    uint64_t fq[4], eq[4], fg[3], eg[3], fvec[2], evec[2];
    uint32_t tmem_base;
    int abort_flag;
};
constexpr uint32_t KV_BARS_BYTES = (sizeof(KvBars) + 255u) & ~255u;
constexpr uint32_t SMEM_MAX = 227u * 1024u;  // dynamic + static shared memory of one CTA

template <int D>
struct BCfg {
    static constexpr int CH = D / 64;
    static constexpr uint32_t TILE = BM * D * 2;
    static constexpr uint32_t RES = 2 * TILE;  // resident pair (K,V) or (Q,dO)
    // Streamed tiles in rings of their own.  The score product of the next
    // tile (S^T(s+1) / S(s+1)) is issued early, but a ring slot is freed only
    // by the last product of the tile it held, so the operand of the score
    // product gets one slot more than the other one.
    // dK/dV kernel: Q ring, dO ring, a two-slot ring of the LSE/delta vectors of
    // the Q tile in work, and the barriers (three Q slots at d = 128: the score
    // product S^T(s+1) is issued while dK(s-1) still reads Q(s-1)).  The tiles
    // start on a 1024-byte boundary; the kernel checks that its layout fits.
    static constexpr int NQS = D == 64 ? 4 : 3;
    static constexpr int NGS = D == 64 ? 3 : 2;
    static constexpr uint32_t KV_NEED = RES + (NQS + NGS) * TILE + 2 * VEC_BYTES + KV_BARS_BYTES;
    static constexpr uint32_t SMEM_KV = KV_NEED + 1024 <= SMEM_MAX ? KV_NEED + 1024 : SMEM_MAX;
    // dQ kernel: K ring, V ring
    static constexpr int NKS = D == 64 ? 4 : 3;
    static constexpr int NVS = D == 64 ? 3 : 2;
    static constexpr uint32_t SMEM_Q = RES + (NKS + NVS) * TILE + 1024;
    // keep one CTA per SM (all 512 tensor-memory columns each)
    static constexpr uint32_t SMEM_KV_REQ = SMEM_KV < 120u * 1024u ? 120u * 1024u : SMEM_KV;
    static constexpr uint32_t SMEM_Q_REQ = SMEM_Q < 120u * 1024u ? 120u * 1024u : SMEM_Q;
    static_assert(KV_NEED <= SMEM_MAX && SMEM_Q <= SMEM_MAX, "backward rings exceed shared memory");
    static_assert(NQS <= 4 && NGS <= 3, "ring depths exceed the barrier arrays");
};

struct BwdParams {
    int N, BH, n_q, pitch;
    int dreal;   // head width of the tensors (<= D: narrower heads are padded with zeros)
    float sl, scale;
    uint64_t limit;
    const float *lse2, *delta;  // [BH][pitch]
    void *dq, *dk, *dv;
    int g_fp32;
    int hgroup;  // causal dQ order: heads per group (see fa_bwd_dq_tc)
};

// Columns 0 .. ncols - 1 of a 32-column chunk (ncols a multiple of 8, <= 32),
// times `mul`.
__device__ __forceinline__ void store_row32(void *base, int fp32, size_t elem, const uint32_t (&raw)[32], float mul,
                                            int ncols = 32)
{
    if (fp32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(base) + elem);
#pragma unroll
        for (int x = 0; x < 8; ++x)
            if (4 * x < ncols) dst[x] = make_float4(__uint_as_float(raw[4 * x]) * mul, __uint_as_float(raw[4 * x + 1]) * mul,
                                 __uint_as_float(raw[4 * x + 2]) * mul, __uint_as_float(raw[4 * x + 3]) * mul);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + elem);
#pragma unroll
        for (int x = 0; x < 4; ++x)
            if (8 * x < ncols) dst[x] = make_uint4(pack_bf16x2(__uint_as_float(raw[8 * x]) * mul, __uint_as_float(raw[8 * x + 1]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * mul, __uint_as_float(raw[8 * x + 3]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * mul, __uint_as_float(raw[8 * x + 5]) * mul),
                                pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * mul, __uint_as_float(raw[8 * x + 7]) * mul));
    }
}

// Tensor-memory column of K step kk (16 elements) of a 128-wide bf16 A
// operand whose W-element column groups were written by the group's warps
// at col0 + g W (W / 2 packed columns each, over the group's own fp32 columns).
template <int W>
__device__ __forceinline__ uint32_t a_col(uint32_t col0, int kk)
{
    const int e = 16 * kk;
    return col0 + (uint32_t)((e / W) * W + (e % W) / 2);
}

// Row slices of tensor memory by width (32 lanes; loads include the wait):
// W fp32 columns in, W / 2 packed bf16 columns out, for W = 32 or 64.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t a, uint32_t (&r)[NC])
{
    static_assert(NC == 32 || NC == 64, "tmem_ld_cols: 32 or 64 columns");
    if constexpr (NC == 32) tmem_ld32(a, r);
    else tmem_ld64(a, r);
}
template <int NC>
__device__ __forceinline__ void tmem_st_cols(uint32_t a, const uint32_t (&r)[NC])
{
    static_assert(NC == 16 || NC == 32, "tmem_st_cols: 16 or 32 columns");
    if constexpr (NC == 16) tmem_st16(a, r);
    else tmem_st32(a, r);
}

constexpr uint32_t ERR_BWD_WAIT = 64u;     // a backward wait gave up (bits distinct from the forward kernels')
constexpr uint32_t ERR_BWD_LAYOUT = 128u;  // the dK/dV kernel's shared-memory layout did not fit its allocation

__device__ __forceinline__ void fail_bwd(volatile int *abort_flag)
{
    atomicOr(&g_bwd_error_word, ERR_BWD_WAIT);
    *abort_flag = 1;
}

// Work item `it` of this CTA: its block index, or (persistent CTAs, short
// items) rounds of alternating direction over the CTAs, so that items of
// unequal length (causal) even out per CTA.
template <bool PERSIST>
__device__ __forceinline__ int bwd_item_index(int it)
{
    if (!PERSIST) return it == 0 ? (int)blockIdx.x : INT_MAX;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    return it * G + ((it & 1) ? G - 1 - c : c);
}

// Slot and phase parity of a ring of N slots at some step, advanced one step
// at a time (no division by N in the issue loops).
struct RingPos {
    int slot;
    uint32_t phase;
};
template <int N>
__device__ __forceinline__ RingPos ring_next(RingPos p)
{
    return p.slot + 1 == N ? RingPos{0, p.phase ^ 1u} : RingPos{p.slot + 1, p.phase};
}

// ---------------------------------------------------------------- dK / dV
// A work item is one 128-key tile of one head.  With PERSIST a CTA loops over
// several: the steps (query tiles) of all its items are numbered globally, so
// the rings and the per-step barriers run on across items; the resident K and
// V of the next item load once the last score products of the current one
// have read theirs (res_empty), and its first dV product waits until the
// epilogue has read the current dV and dK from tensor memory (acc_empty).
template <int D, bool CAUSAL, bool PERSIST>
__global__ void __launch_bounds__(EW<D>::NUM_THREADS, 1)
fa_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g, const BwdParams prm)
{
    using C = BCfg<D>;
    using E = EW<D>;
    constexpr int W = E::W, TMA_WARP = E::TMA_WARP, MMA_WARP = E::MMA_WARP;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N;
    const int n_items = prm.n_q * prm.BH;
    // item it: key tile kt of head bh, query tiles first .. n_q - 1
    auto item = [&](int it, int &k0, int &bh, int &first, int &n_steps) -> bool {
        const int w = bwd_item_index<PERSIST>(it);
        if (w >= n_items) return false;
        const int kt = w % prm.n_q;
        bh = w / prm.n_q;
        k0 = kt * BM;
        first = CAUSAL ? kt : 0;  // query tiles before the key tile see none of its keys
        n_steps = prm.n_q - first;
        return true;
    };

    // 1024-byte aligned base, derived from smem_raw by an offset so the
    // compiler keeps the shared address space (plain shared loads for the
    // per-query vectors).  The layout must fit the allocation (it does when the
    // allocation starts within a few hundred bytes of a 1024-byte boundary, as
    // a CTA's shared memory does without static shared variables): checked here,
    // with every thread leaving before any barrier or tensor memory is touched.
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    if (pad + C::KV_NEED > C::SMEM_KV_REQ) {
        if (threadIdx.x == 0) atomicOr(&g_bwd_error_word, ERR_BWD_LAYOUT);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    const uint32_t s_base = smem_addr(smem);
    const uint32_t sK = s_base, sV = s_base + C::TILE;
    // Q ring, dO ring, the vector ring (LSE * log2 e, then delta, of 128 queries
    // per slot), the barriers
    const uint32_t sQr = s_base + C::RES, sGr = sQr + C::NQS * C::TILE;
    const uint32_t oVec = C::RES + (C::NQS + C::NGS) * C::TILE;
    KvBars &bars = *reinterpret_cast<KvBars *>(smem + C::KV_NEED - KV_BARS_BYTES);
    // per ring slot: fq/eq for Q_i, fg/eg for dO_i (dO_i is freed by the earlier dV
    // product and loaded second, so Q_i, needed first, lands sooner), fvec/evec for
    // the vectors of the step in work (freed by the elementwise warps)
    uint64_t &res_full = bars.res_full, &res_empty = bars.res_empty, &st_full = bars.st_full, &s_read = bars.s_read,
             &dp_full = bars.dp_full, &p_ready = bars.p_ready, &ds_ready = bars.ds_ready, &o_full = bars.o_full,
             &acc_empty = bars.acc_empty, &drain = bars.drain;
    uint64_t *fq = bars.fq, *eq = bars.eq, *fg = bars.fg, *eg = bars.eg, *fvec = bars.fvec, *evec = bars.evec;
    volatile int &abort_flag = *const_cast<volatile int *>(&bars.abort_flag);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&res_full), 1);
        mbar_init(smem_addr(&res_empty), 1);
        for (int s = 0; s < C::NQS; ++s) {
            mbar_init(smem_addr(&fq[s]), 1);
            mbar_init(smem_addr(&eq[s]), 1);
        }
        for (int s = 0; s < C::NGS; ++s) {
            mbar_init(smem_addr(&fg[s]), 1);
            mbar_init(smem_addr(&eg[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_addr(&fvec[s]), 1);
            mbar_init(smem_addr(&evec[s]), E::THREADS);
        }
        mbar_init(smem_addr(&st_full), 1);
        mbar_init(smem_addr(&s_read), E::THREADS);
        mbar_init(smem_addr(&dp_full), 1);
        mbar_init(smem_addr(&p_ready), E::THREADS);
        mbar_init(smem_addr(&ds_ready), E::THREADS);
        mbar_init(smem_addr(&o_full), 1);
        mbar_init(smem_addr(&acc_empty), E::THREADS);
        mbar_init(smem_addr(&drain), 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(&bars.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the dQ kernel (independent of this one) may take SMs as this grid's last
    // CTAs leave them
    pdl_launch_dependents();
    const uint32_t tmem = bars.tmem_base;
    const uint64_t limit = prm.limit;
    // tensor memory: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D, 256+2D).
    // Once the elementwise warps hold dP^T(s) in registers, the column half h
    // of P^T(s) goes to columns [128 + 64h, +32) and of dS^T(s) to [128 + 64h + 32,
    // +32), over the dP^T values that half has read: the S^T columns are free
    // as soon as S^T(s) is in registers, so S^T(s+1) runs while they work on s.
    const uint32_t cS = 0, cP = 128, cV = 256, cK = 256 + D;

    if (warp == TMA_WARP) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            bool ok = true;
            int g = 0;  // global step: ring positions run on across items
            int issued_q = 0, issued_g = 0, issued_v = 0, res_items = 0;
            int k0, bh, first, n_steps;
            bool have = item(0, k0, bh, first, n_steps);
            for (int it = 0; ok && have; ++it) {
                // the item's resident K and V, once the previous item's are read: the
                // first item's before anything else, a later one's after the first
                // step's Q and vectors (which need not wait for them)
                auto load_res = [&]() -> bool {
                    if (it > 0 && !wait_or_abort(smem_addr(&res_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag))
                        return false;
                    mbar_arrive_expect_tx(smem_addr(&res_full), C::RES);
                    for (int c = 0; c < C::CH; ++c) {
                        tma_load_3d(sK + c * BOX, &tm_k, smem_addr(&res_full), c * 64, k0, bh, pol);
                        tma_load_3d(sV + c * BOX, &tm_v, smem_addr(&res_full), c * 64, k0, bh, pol);
                    }
                    res_items = it + 1;
                    return true;
                };
                if (it == 0 && !(ok = load_res())) break;
                for (int s = 0; s < n_steps; ++s, ++g) {
                    const int qs = g % C::NQS, gs = g % C::NGS, vs = g & 1, q0 = (first + s) * BM;
                    if (!wait_or_abort(smem_addr(&eq[qs]), (uint32_t)(((g / C::NQS) & 1) ^ 1), limit, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bq = smem_addr(&fq[qs]);
                    mbar_arrive_expect_tx(bq, C::TILE);
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_3d(sQr + qs * C::TILE + c * BOX, &tm_q, bq, c * 64, q0, bh, pol);
                    issued_q = g + 1;
                    if (!wait_or_abort(smem_addr(&evec[vs]), (uint32_t)(((g >> 1) & 1) ^ 1), limit, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bv = smem_addr(&fvec[vs]);
                    mbar_arrive_expect_tx(bv, VEC_BYTES);
                    const size_t vrow = (size_t)bh * prm.pitch + q0;
                    const uint32_t dvec = s_base + oVec + vs * VEC_BYTES;
                    bulk_copy_g2s(dvec, prm.lse2 + vrow, 512, bv);
                    bulk_copy_g2s(dvec + 512, prm.delta + vrow, 512, bv);
                    issued_v = g + 1;
                    if (s == 0 && it > 0 && !(ok = load_res())) break;
                    if (!wait_or_abort(smem_addr(&eg[gs]), (uint32_t)(((g / C::NGS) & 1) ^ 1), limit, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bg = smem_addr(&fg[gs]);
                    mbar_arrive_expect_tx(bg, C::TILE);
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_3d(sGr + gs * C::TILE + c * BOX, &tm_g, bg, c * 64, q0, bh, pol);
                    issued_g = g + 1;
                }
                if constexpr (!PERSIST) break;  // one item per CTA
                have = item(it + 1, k0, bh, first, n_steps);
            }
            if (!ok) {
                if (!abort_flag) fail_bwd(&abort_flag);
                for (int x = (issued_q > C::NQS ? issued_q - C::NQS : 0); x < issued_q; ++x)
                    mbar_wait_bounded(smem_addr(&fq[x % C::NQS]), (uint32_t)((x / C::NQS) & 1), limit);
                for (int x = (issued_v > 2 ? issued_v - 2 : 0); x < issued_v; ++x)
                    mbar_wait_bounded(smem_addr(&fvec[x & 1]), (uint32_t)((x >> 1) & 1), limit);
                for (int x = (issued_g > C::NGS ? issued_g - C::NGS : 0); x < issued_g; ++x)
                    mbar_wait_bounded(smem_addr(&fg[x % C::NGS]), (uint32_t)((x / C::NGS) & 1), limit);
                if (res_items > 0) mbar_wait_bounded(smem_addr(&res_full), (uint32_t)((res_items - 1) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        {  // whole warp, converged; elect.sync picks the issuing lane
            const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0), id_o = idesc_bf16_f32(BM, D, 0, 1);
            const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
            bool ok = true, issued = false;
            // S^T(g) = K Q_g^T into cS, dP^T(g) = V dO_g^T into cP (g a global step;
            // the _at forms take the ring slot)
            auto mma_st_at = [&](int slot) {
                const uint64_t dQ = sdesc_sw128(sQr + slot * C::TILE, 16, 1024);
                uint64_t ka[D / 16], kb[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * BOX + (kk & 3) * 32) >> 4);
                    ka[kk] = dK + off;
                    kb[kk] = dQ + off;
                }
                mma_ss_k<D / 16>(tmem + cS, ka, kb, id_s, 0u);
                issued = true;
            };
            auto mma_dpt_at = [&](int slot) {
                const uint64_t dG = sdesc_sw128(sGr + slot * C::TILE, 16, 1024);
                uint64_t ka[D / 16], kb[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * BOX + (kk & 3) * 32) >> 4);
                    ka[kk] = dV + off;
                    kb[kk] = dG + off;
                }
                mma_ss_k<D / 16>(tmem + cP, ka, kb, id_s, 0u);
            };
            auto mma_st = [&](int g) { mma_st_at(g % C::NQS); };
            auto mma_dpt = [&](int g) { mma_dpt_at(g % C::NGS); };
            // dV += P^T dO_g (A: the P^T columns of cP) or dK += dS^T Q_g (A: the
            // dS^T columns, 32 further), B MN-major from its ring slot; the first
            // step of an item overwrites
            auto mma_acc = [&](uint32_t d_col, uint32_t a_col0, uint64_t b_mn, int s) {
                uint32_t ta[BM / 16];
                uint64_t tb[BM / 16];
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    ta[kk] = tmem + a_col<W>(a_col0, kk);
                    tb[kk] = b_mn + (uint64_t)((kk * 16 * 128) >> 4);
                }
                mma_ts_k<BM / 16>(tmem + d_col, ta, tb, id_o, s > 0 ? 1u : 0u);
            };
            // Q_g in ring slot g % NQS, dO_g in slot g % NGS
            auto wait_at = [&](uint64_t *full, RingPos p) -> bool {
                if (!wait_or_abort_w(smem_addr(&full[p.slot]), p.phase, limit, &abort_flag)) return false;
                tc_fence_after();
                return true;
            };
            auto wait_q = [&](int g) { return wait_at(fq, RingPos{g % C::NQS, (uint32_t)((g / C::NQS) & 1)}); };
            auto wait_g = [&](int g) { return wait_at(fg, RingPos{g % C::NGS, (uint32_t)((g / C::NGS) & 1)}); };
            if constexpr (!PERSIST) {
                // One item.  (The item loop below, run for one item, measured 4 %
                // slower on long sequences than this plain loop.)
                int k0, bh, first, n_steps;
                item(0, k0, bh, first, n_steps);
                ok = wait_or_abort_w(smem_addr(&res_full), 0, limit, &abort_flag);
                if (ok && (ok = wait_q(0))) {
                    mma_st(0);
                    mma_commit_w(smem_addr(&st_full));
                    if ((ok = wait_g(0))) {
                        mma_dpt(0);
                        mma_commit_w(smem_addr(&dp_full));
                    }
                }
                // Per step: S^T(s+1) once the elementwise warps hold S^T(s) (it runs while
                // they compute the weights of step s); dV(s) once P^T(s) is written; dK(s)
                // once dS^T(s) is; then dP^T(s+1) over the columns those two have read.
                for (int s = 0; ok && s < n_steps; ++s) {
                    const bool more = s + 1 < n_steps;
                    if (more) {
                        if (!wait_or_abort_w(smem_addr(&s_read), (uint32_t)(s & 1), limit, &abort_flag) || !wait_q(s + 1)) {
                            ok = false;
                            break;
                        }
                        mma_st(s + 1);
                        mma_commit_w(smem_addr(&st_full));
                    }
                    if (!wait_or_abort_w(smem_addr(&p_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    mma_acc(cV, cP, sdesc_sw128(sGr + (s % C::NGS) * C::TILE, BOX, 1024), s);
                    mma_commit_w(smem_addr(&eg[s % C::NGS]));  // dO_s read for the last time
                    if (!wait_or_abort_w(smem_addr(&ds_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    mma_acc(cK, cP + W / 2, sdesc_sw128(sQr + (s % C::NQS) * C::TILE, BOX, 1024), s);
                    mma_commit_w(smem_addr(&eq[s % C::NQS]));  // Q_s read for the last time
                    if (more) {
                        if (!wait_g(s + 1)) { ok = false; break; }
                        mma_dpt(s + 1);
                        mma_commit_w(smem_addr(&dp_full));
                    }
                }
                if (ok) mma_commit_w(smem_addr(&o_full));
            } else {
                // Items one after the other, steps numbered globally.  An item's first
                // two score products wait for its resident K and V (and for the
                // previous S^T to be in registers); its first dV product waits until
                // the previous item's dV and dK have left tensor memory.
                RingPos q{0, 0u}, gq{0, 0u};  // Q and dO ring positions of the step in work
                uint32_t par = 0;              // parity of the step in work (per-step barriers)
                int k0, bh, first, n_steps;
                bool have = item(0, k0, bh, first, n_steps);
                for (int it = 0; ok && have; ++it) {
                    if (!wait_or_abort_w(smem_addr(&res_full), (uint32_t)(it & 1), limit, &abort_flag) ||
                        (it > 0 && !wait_or_abort_w(smem_addr(&s_read), par ^ 1u, limit, &abort_flag)) ||
                        !wait_at(fq, q)) {
                        ok = false;
                        break;
                    }
                    mma_st_at(q.slot);
                    mma_commit_w(smem_addr(&st_full));
                    if (!wait_at(fg, gq)) { ok = false; break; }
                    mma_dpt_at(gq.slot);
                    mma_commit_w(smem_addr(&dp_full));
                    if (n_steps == 1) mma_commit_w(smem_addr(&res_empty));  // K and V read for the last time
                    for (int s = 0; s < n_steps; ++s) {
                        const bool more = s + 1 < n_steps;
                        const RingPos q1 = ring_next<C::NQS>(q), gq1 = ring_next<C::NGS>(gq);
                        if (more) {
                            if (!wait_or_abort_w(smem_addr(&s_read), par, limit, &abort_flag) || !wait_at(fq, q1)) {
                                ok = false;
                                break;
                            }
                            mma_st_at(q1.slot);
                            mma_commit_w(smem_addr(&st_full));
                        }
                        if (!wait_or_abort_w(smem_addr(&p_ready), par, limit, &abort_flag) ||
                            (s == 0 && it > 0 &&
                             !wait_or_abort_w(smem_addr(&acc_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_acc(cV, cP, sdesc_sw128(sGr + gq.slot * C::TILE, BOX, 1024), s);
                        mma_commit_w(smem_addr(&eg[gq.slot]));  // dO of this step read for the last time
                        if (!wait_or_abort_w(smem_addr(&ds_ready), par, limit, &abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        mma_acc(cK, cP + W / 2, sdesc_sw128(sQr + q.slot * C::TILE, BOX, 1024), s);
                        mma_commit_w(smem_addr(&eq[q.slot]));  // Q of this step read for the last time
                        if (more) {
                            if (!wait_at(fg, gq1)) { ok = false; break; }
                            mma_dpt_at(gq1.slot);
                            mma_commit_w(smem_addr(&dp_full));
                            if (s + 2 == n_steps) mma_commit_w(smem_addr(&res_empty));  // K and V read for the last time
                        }
                        q = q1;
                        gq = gq1;
                        par ^= 1u;
                    }
                    if (!ok) break;
                    mma_commit_w(smem_addr(&o_full));  // this item's dV and dK are complete
                    have = item(it + 1, k0, bh, first, n_steps);
                }
            }
            if (!ok) {
                if (!abort_flag) fail_bwd(&abort_flag);
                if (issued) {
                    mma_commit_w(smem_addr(&drain));
                    mbar_wait_bounded(smem_addr(&drain), 0, limit);
                }
            }
        }
        __syncwarp();
    } else {
        // one key per thread (tensor-memory lane), queries [W hf, W hf + W) of each tile
        const int quarter = warp & 3, hf = warp >> 2;
        const int jr = quarter * 32 + lane;
        const uint32_t lb = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t cSh = cS + hf * W, cPh = cP + hf * W;
        const float sl = prm.sl;
        bool ok = true;
        int g = 0;
        int k0, bh, first, n_steps;
        bool have = item(0, k0, bh, first, n_steps);
        for (int it = 0; ok && have; ++it) {
            const int kj = k0 + jr;
            for (int s = 0; s < n_steps; ++s, ++g) {
                const int vs = g & 1, q0 = (first + s) * BM + hf * W;
                if (!wait_or_abort(smem_addr(&st_full), (uint32_t)(g & 1), limit, &abort_flag) ||
                    !wait_or_abort(smem_addr(&fvec[vs]), (uint32_t)((g >> 1) & 1), limit, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float4 *vec = reinterpret_cast<const float4 *>(smem + oVec + vs * VEC_BYTES) + hf * (W / 4);
                // Tiles with no padded key or query and wholly below the diagonal
                // take the unmasked path (no per-element tests or selects).
                const int qt0 = (first + s) * BM;
                const bool masked = k0 + BM > N || qt0 + BM > N || (CAUSAL && qt0 < k0 + BM);
                // P^T row: weights of this key for this half of the tile's queries, as
                // bf16 pairs (kept in registers for dS^T, written to tensor memory for
                // the dV product once dP^T(s) has been read)
                uint32_t pw[W / 2];
                {
                    uint32_t raw[W];
                    tmem_ld_cols(lb + cSh, raw);
                    tc_fence_before();
                    mbar_arrive(smem_addr(&s_read));  // S^T(s) is in registers: S^T(s+1) may overwrite it
                    const uint64_t sl2 = f2_pack(sl, sl);
                    auto weights = [&](auto mask) {
                        constexpr bool M = decltype(mask)::value;
#pragma unroll
                        for (int c4 = 0; c4 < W / 4; ++c4) {
                            const float4 l4 = vec[c4];  // LSE * log2 e of queries q0 + 4 c4 ...
#pragma unroll
                            for (int e = 0; e < 4; e += 2) {
                                const int c = 4 * c4 + e;
                                const uint64_t nl = e ? f2_pack(-l4.z, -l4.w) : f2_pack(-l4.x, -l4.y);
                                float a0, a1;
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), sl2, nl), a0, a1);
                                float w0 = ex2(a0), w1 = ex2(a1);
                                if (M) {
                                    const int q = q0 + c;
                                    w0 = (kj < N && q < N && (!CAUSAL || kj <= q)) ? w0 : 0.f;
                                    w1 = (kj < N && q + 1 < N && (!CAUSAL || kj <= q + 1)) ? w1 : 0.f;
                                }
                                pw[c / 2] = pack_bf16x2(w0, w1);
                            }
                        }
                    };
                    if (masked) weights(std::true_type{});
                    else weights(std::false_type{});
                }
                // dP^T(s) into registers; its columns then take P^T (for dV) and dS^T
                // = P^T (dP^T - delta), with the bf16 weights the dV product uses
                if (!wait_or_abort(smem_addr(&dp_full), (uint32_t)(g & 1), limit, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t raw[W];
                    tmem_ld_cols(lb + cPh, raw);
                    tmem_st_cols(lb + cPh, pw);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_addr(&p_ready));
                    uint32_t pk[W / 2];
                    // a masked weight is exactly 0 and its dP may be anything, so the
                    // masked path selects 0 instead of multiplying
                    auto grads = [&](auto mask) {
                        constexpr bool M = decltype(mask)::value;
#pragma unroll
                        for (int c4 = 0; c4 < W / 4; ++c4) {
                            const float4 d4 = vec[BM / 4 + c4];  // delta of queries q0 + 4 c4 ...
#pragma unroll
                            for (int e = 0; e < 4; e += 2) {
                                const int c = 4 * c4 + e;
                                const uint64_t nd = e ? f2_pack(-d4.z, -d4.w) : f2_pack(-d4.x, -d4.y);
                                const float p0 = __uint_as_float(pw[c / 2] << 16), p1 = __uint_as_float(pw[c / 2] & 0xffff0000u);
                                const uint64_t t = f2_add(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), nd);
                                float d0, d1;
                                f2_unpack(f2_mul(f2_pack(p0, p1), t), d0, d1);
                                if (M) {
                                    d0 = p0 != 0.f ? d0 : 0.f;
                                    d1 = p1 != 0.f ? d1 : 0.f;
                                }
                                pk[c / 2] = pack_bf16x2(d0, d1);
                            }
                        }
                    };
                    if (masked) grads(std::true_type{});
                    else grads(std::false_type{});
                    mbar_arrive(smem_addr(&evec[vs]));  // this step's vectors are read
                    tmem_st_cols(lb + cPh + W / 2, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_addr(&ds_ready));
            }
            if (!ok || !wait_or_abort(smem_addr(&o_full), (uint32_t)(it & 1), limit, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const size_t row = ((size_t)bh * N + kj) * prm.dreal;
#pragma unroll 1
            for (int c = hf; c < D / 32; c += E::NH) {  // this warp's 32-column chunks
                uint32_t raw[32];
                const int nc = min(32, prm.dreal - c * 32);  // a padded head stores its own columns only
                tmem_ld32(lb + cV + c * 32, raw);
                if (kj < N && nc > 0) store_row32(prm.dv, prm.g_fp32, row + c * 32, raw, 1.f, nc);
                tmem_ld32(lb + cK + c * 32, raw);
                if (kj < N && nc > 0) store_row32(prm.dk, prm.g_fp32, row + c * 32, raw, prm.scale, nc);
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&acc_empty));  // dV and dK read: the next item may overwrite them
            if constexpr (!PERSIST) break;  // one item per CTA
            have = item(it + 1, k0, bh, first, n_steps);
        }
        if (!ok && !abort_flag) fail_bwd(&abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- dQ
// A work item is one 128-query tile of one head; PERSIST as in the dK/dV
// kernel, with the resident Q and dO and the accumulator dQ handed over
// between items by res_empty and acc_empty.
template <int D, bool CAUSAL, bool PERSIST>
__global__ void __launch_bounds__(EW<D>::NUM_THREADS, 1)
fa_bwd_dq_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g, const BwdParams prm)
{
    using C = BCfg<D>;
    using E = EW<D>;
    constexpr int W = E::W, TMA_WARP = E::TMA_WARP, MMA_WARP = E::MMA_WARP;
    extern __shared__ uint8_t smem_raw[];
    // per ring slot: fk/ek for K_j, fv/ev for V_j (V_j is freed by the earlier dP
    // product and loaded second, so K_j, needed first, lands sooner)
    __shared__ __align__(8) uint64_t res_full, res_empty, fk[C::NKS], ek[C::NKS], fv[C::NVS], ev[C::NVS], s_full,
        dp_full, s_read, ds_ready, o_full, acc_empty, drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N;
    const int n_items = prm.n_q * prm.BH;
    // item it: query tile qt of head bh, key tiles 0 .. n_steps - 1.  Causal:
    // heads in groups of hgroup whose K and V fit in L2 together, one group
    // after the other, the longest query tiles of a group first
    auto item = [&](int it, int &q0, int &bh, int &n_steps) -> bool {
        const int w = bwd_item_index<PERSIST>(it);
        if (w >= n_items) return false;
        int qt;
        if (CAUSAL) {
            const int per = prm.hgroup * prm.n_q;
            const int g0 = (w / per) * prm.hgroup, x = w % per;
            const int gh = min(prm.hgroup, prm.BH - g0);
            qt = prm.n_q - 1 - x / gh;
            bh = g0 + x % gh;
        } else {
            qt = w % prm.n_q;
            bh = w / prm.n_q;
        }
        q0 = qt * BM;
        n_steps = CAUSAL ? qt + 1 : prm.n_q;  // key tiles this query tile sees
        return true;
    };

    // 1024-byte aligned base, derived from smem_raw by an offset so the
    // compiler keeps the shared address space (plain shared loads for the
    // per-query vectors)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t s_base = smem_addr(smem);
    const uint32_t sQ = s_base, sG = s_base + C::TILE;
    const uint32_t sKr = s_base + C::RES, sVr = sKr + C::NKS * C::TILE;  // K ring, V ring

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&res_full), 1);
        mbar_init(smem_addr(&res_empty), 1);
        for (int s = 0; s < C::NKS; ++s) {
            mbar_init(smem_addr(&fk[s]), 1);
            mbar_init(smem_addr(&ek[s]), 1);
        }
        for (int s = 0; s < C::NVS; ++s) {
            mbar_init(smem_addr(&fv[s]), 1);
            mbar_init(smem_addr(&ev[s]), 1);
        }
        mbar_init(smem_addr(&s_full), 1);
        mbar_init(smem_addr(&dp_full), 1);
        mbar_init(smem_addr(&s_read), E::THREADS);
        mbar_init(smem_addr(&ds_ready), E::THREADS);
        mbar_init(smem_addr(&o_full), 1);
        mbar_init(smem_addr(&acc_empty), E::THREADS);
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
    const uint64_t limit = prm.limit;
    // tensor memory: S [0,128), dP / dS [128,256), dQ [256, 256+D); the column half h
    // of dS is written over columns [64h, 64h + 32) of dP
    const uint32_t cS = 0, cP = 128, cQ = 256;

    if (warp == TMA_WARP) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            bool ok = true;
            int g = 0;  // global step: ring positions run on across items
            int issued_k = 0, issued_v = 0, res_items = 0;
            int q0, bh, n_steps;
            bool have = item(0, q0, bh, n_steps);
            for (int it = 0; ok && have; ++it) {
                // the item's resident Q and dO, once the previous item's are read: the
                // first item's before anything else, a later one's after the first
                // step's K (which need not wait for them)
                auto load_res = [&]() -> bool {
                    if (it > 0 && !wait_or_abort(smem_addr(&res_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag))
                        return false;
                    mbar_arrive_expect_tx(smem_addr(&res_full), C::RES);
                    for (int c = 0; c < C::CH; ++c) {
                        tma_load_3d(sQ + c * BOX, &tm_q, smem_addr(&res_full), c * 64, q0, bh, pol);
                        tma_load_3d(sG + c * BOX, &tm_g, smem_addr(&res_full), c * 64, q0, bh, pol);
                    }
                    res_items = it + 1;
                    return true;
                };
                if (it == 0 && !(ok = load_res())) break;
                for (int s = 0; s < n_steps; ++s, ++g) {
                    const int ks = g % C::NKS, vs = g % C::NVS, k0 = s * BM;
                    if (!wait_or_abort(smem_addr(&ek[ks]), (uint32_t)(((g / C::NKS) & 1) ^ 1), limit, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bk = smem_addr(&fk[ks]);
                    mbar_arrive_expect_tx(bk, C::TILE);
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_3d(sKr + ks * C::TILE + c * BOX, &tm_k, bk, c * 64, k0, bh, pol);
                    issued_k = g + 1;
                    if (s == 0 && it > 0 && !(ok = load_res())) break;
                    if (!wait_or_abort(smem_addr(&ev[vs]), (uint32_t)(((g / C::NVS) & 1) ^ 1), limit, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bv = smem_addr(&fv[vs]);
                    mbar_arrive_expect_tx(bv, C::TILE);
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_3d(sVr + vs * C::TILE + c * BOX, &tm_v, bv, c * 64, k0, bh, pol);
                    issued_v = g + 1;
                }
                if constexpr (!PERSIST) break;  // one item per CTA
                have = item(it + 1, q0, bh, n_steps);
            }
            if (!ok) {
                if (!abort_flag) fail_bwd(&abort_flag);
                for (int x = (issued_k > C::NKS ? issued_k - C::NKS : 0); x < issued_k; ++x)
                    mbar_wait_bounded(smem_addr(&fk[x % C::NKS]), (uint32_t)((x / C::NKS) & 1), limit);
                for (int x = (issued_v > C::NVS ? issued_v - C::NVS : 0); x < issued_v; ++x)
                    mbar_wait_bounded(smem_addr(&fv[x % C::NVS]), (uint32_t)((x / C::NVS) & 1), limit);
                if (res_items > 0) mbar_wait_bounded(smem_addr(&res_full), (uint32_t)((res_items - 1) & 1), limit);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        {  // whole warp, converged; elect.sync picks the issuing lane
            const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0), id_o = idesc_bf16_f32(BM, D, 0, 1);
            const uint64_t dQ = sdesc_sw128(sQ, 16, 1024), dG = sdesc_sw128(sG, 16, 1024);
            bool ok = true, issued = false;
            // K_g in ring slot g % NKS, V_g in slot g % NVS (g a global step; the _at
            // forms take the ring slot)
            auto wait_at = [&](uint64_t *full, RingPos p) -> bool {
                if (!wait_or_abort_w(smem_addr(&full[p.slot]), p.phase, limit, &abort_flag)) return false;
                tc_fence_after();
                return true;
            };
            auto wait_k = [&](int g) { return wait_at(fk, RingPos{g % C::NKS, (uint32_t)((g / C::NKS) & 1)}); };
            auto wait_v = [&](int g) { return wait_at(fv, RingPos{g % C::NVS, (uint32_t)((g / C::NVS) & 1)}); };
            // S(g) = Q K_g^T into cS; dP(g) = dO V_g^T into cP
            auto mma_s_at = [&](int slot) {
                const uint64_t dK = sdesc_sw128(sKr + slot * C::TILE, 16, 1024);
                uint64_t ka[D / 16], kb[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * BOX + (kk & 3) * 32) >> 4);
                    ka[kk] = dQ + off;
                    kb[kk] = dK + off;
                }
                mma_ss_k<D / 16>(tmem + cS, ka, kb, id_s, 0u);
                issued = true;
            };
            auto mma_dp_at = [&](int slot) {
                const uint64_t dV = sdesc_sw128(sVr + slot * C::TILE, 16, 1024);
                uint64_t ka[D / 16], kb[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * BOX + (kk & 3) * 32) >> 4);
                    ka[kk] = dG + off;
                    kb[kk] = dV + off;
                }
                mma_ss_k<D / 16>(tmem + cP, ka, kb, id_s, 0u);
            };
            auto mma_s = [&](int g) { mma_s_at(g % C::NKS); };
            auto mma_dp = [&](int g) { mma_dp_at(g % C::NVS); };
            // dQ += dS K (A: dS over the dP columns, B: the K tile of ring slot
            // `slot`, MN-major); the first step of an item overwrites
            auto mma_dq = [&](int slot, int s) {
                const uint64_t dKmn = sdesc_sw128(sKr + slot * C::TILE, BOX, 1024);
                uint32_t ta[BM / 16];
                uint64_t tb[BM / 16];
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    ta[kk] = tmem + a_col<W>(cP, kk);
                    tb[kk] = dKmn + (uint64_t)((kk * 16 * 128) >> 4);
                }
                mma_ts_k<BM / 16>(tmem + cQ, ta, tb, id_o, s > 0 ? 1u : 0u);
            };
            if constexpr (!PERSIST) {
                // One item.  (The item loop below, run for one item, measured 4 %
                // slower on long sequences than this plain loop.)
                int q0, bh, n_steps;
                item(0, q0, bh, n_steps);
                ok = wait_or_abort_w(smem_addr(&res_full), 0, limit, &abort_flag);
                if (ok && (ok = wait_k(0))) {
                    mma_s(0);
                    mma_commit_w(smem_addr(&s_full));
                    if ((ok = wait_v(0))) {
                        mma_dp(0);
                        mma_commit_w(smem_addr(&dp_full));
                        mma_commit_w(smem_addr(&ev[0]));  // V_0 read for the last time
                    }
                }
                // Per step: S(s+1) as soon as the softmax warps have read S(s) (it
                // overlaps their dS(s)); dQ(s) once dS(s) is written over dP(s);
                // then dP(s+1) into the columns dQ(s) has just read.
                for (int s = 0; ok && s < n_steps; ++s) {
                    const bool more = s + 1 < n_steps;
                    if (more) {
                        if (!wait_or_abort_w(smem_addr(&s_read), (uint32_t)(s & 1), limit, &abort_flag) || !wait_k(s + 1)) {
                            ok = false;
                            break;
                        }
                        mma_s(s + 1);
                        mma_commit_w(smem_addr(&s_full));
                    }
                    if (!wait_or_abort_w(smem_addr(&ds_ready), (uint32_t)(s & 1), limit, &abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    mma_dq(s % C::NKS, s);
                    mma_commit_w(smem_addr(&ek[s % C::NKS]));  // K_s read for the last time
                    if (more) {
                        if (!wait_v(s + 1)) { ok = false; break; }
                        mma_dp(s + 1);
                        mma_commit_w(smem_addr(&dp_full));
                        mma_commit_w(smem_addr(&ev[(s + 1) % C::NVS]));  // V_(s+1) read for the last time
                    }
                }
                if (ok) mma_commit_w(smem_addr(&o_full));
            } else {
                // Items one after the other, steps numbered globally, handed over as
                // in the dK/dV kernel (res_full / res_empty, acc_empty).
                RingPos kq{0, 0u}, vq{0, 0u};  // K and V ring positions of the step in work
                uint32_t par = 0;              // parity of the step in work (per-step barriers)
                int q0, bh, n_steps;
                bool have = item(0, q0, bh, n_steps);
                for (int it = 0; ok && have; ++it) {
                    if (!wait_or_abort_w(smem_addr(&res_full), (uint32_t)(it & 1), limit, &abort_flag) ||
                        (it > 0 && !wait_or_abort_w(smem_addr(&s_read), par ^ 1u, limit, &abort_flag)) ||
                        !wait_at(fk, kq)) {
                        ok = false;
                        break;
                    }
                    mma_s_at(kq.slot);
                    mma_commit_w(smem_addr(&s_full));
                    if (!wait_at(fv, vq)) { ok = false; break; }
                    mma_dp_at(vq.slot);
                    mma_commit_w(smem_addr(&dp_full));
                    mma_commit_w(smem_addr(&ev[vq.slot]));  // this V tile read for the last time
                    if (n_steps == 1) mma_commit_w(smem_addr(&res_empty));  // Q and dO read for the last time
                    for (int s = 0; s < n_steps; ++s) {
                        const bool more = s + 1 < n_steps;
                        const RingPos kq1 = ring_next<C::NKS>(kq), vq1 = ring_next<C::NVS>(vq);
                        if (more) {
                            if (!wait_or_abort_w(smem_addr(&s_read), par, limit, &abort_flag) || !wait_at(fk, kq1)) {
                                ok = false;
                                break;
                            }
                            mma_s_at(kq1.slot);
                            mma_commit_w(smem_addr(&s_full));
                        }
                        if (!wait_or_abort_w(smem_addr(&ds_ready), par, limit, &abort_flag) ||
                            (s == 0 && it > 0 &&
                             !wait_or_abort_w(smem_addr(&acc_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_dq(kq.slot, s);
                        mma_commit_w(smem_addr(&ek[kq.slot]));  // this K tile read for the last time
                        if (more) {
                            if (!wait_at(fv, vq1)) { ok = false; break; }
                            mma_dp_at(vq1.slot);
                            mma_commit_w(smem_addr(&dp_full));
                            mma_commit_w(smem_addr(&ev[vq1.slot]));  // the next V tile read for the last time
                            if (s + 2 == n_steps) mma_commit_w(smem_addr(&res_empty));  // Q and dO read for the last time
                        }
                        kq = kq1;
                        vq = vq1;
                        par ^= 1u;
                    }
                    if (!ok) break;
                    mma_commit_w(smem_addr(&o_full));  // this item's dQ is complete
                    have = item(it + 1, q0, bh, n_steps);
                }
            }
            if (!ok) {
                if (!abort_flag) fail_bwd(&abort_flag);
                if (issued) {
                    mma_commit_w(smem_addr(&drain));
                    mbar_wait_bounded(smem_addr(&drain), 0, limit);
                }
            }
        }
        __syncwarp();
    } else {
        // one query per thread (tensor-memory lane), keys [W hf, W hf + W) of each tile
        const int quarter = warp & 3, hf = warp >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lb = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t cSh = cS + hf * W, cPh = cP + hf * W;
        const float sl = prm.sl;
        bool ok = true;
        int g = 0;
        int q0, bh, n_steps;
        bool have = item(0, q0, bh, n_steps);
        for (int it = 0; ok && have; ++it) {
            const int qi = q0 + r;
            const float l2 = qi < N ? prm.lse2[(size_t)bh * prm.pitch + qi] : 0.f;
            const float de = qi < N ? prm.delta[(size_t)bh * prm.pitch + qi] : 0.f;
            for (int s = 0; s < n_steps; ++s, ++g) {
                const int k0 = s * BM + hf * W;
                if (!wait_or_abort(smem_addr(&s_full), (uint32_t)(g & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                // Tiles with no padded key or query and wholly below the diagonal
                // take the unmasked path (no per-element tests or selects).
                const int kt0 = s * BM;
                const bool masked = kt0 + BM > N || q0 + BM > N || (CAUSAL && kt0 + BM > q0);
                float p[W];
                {
                    uint32_t raw[W];
                    tmem_ld_cols(lb + cSh, raw);
                    tc_fence_before();
                    mbar_arrive(smem_addr(&s_read));  // S(s) is in registers: the MMA may overwrite it
                    const uint64_t sl2 = f2_pack(sl, sl), nl2 = f2_pack(-l2, -l2);
                    auto weights = [&](auto mask) {
                        constexpr bool M = decltype(mask)::value;
#pragma unroll
                        for (int c = 0; c < W; c += 2) {
                            float a0, a1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), sl2, nl2), a0, a1);
                            const float w0 = ex2(a0), w1 = ex2(a1);
                            if (M) {
                                const int kj = k0 + c;
                                p[c] = (qi < N && kj < N && (!CAUSAL || kj <= qi)) ? w0 : 0.f;
                                p[c + 1] = (qi < N && kj + 1 < N && (!CAUSAL || kj + 1 <= qi)) ? w1 : 0.f;
                            } else {
                                p[c] = w0;
                                p[c + 1] = w1;
                            }
                        }
                    };
                    if (masked) weights(std::true_type{});
                    else weights(std::false_type{});
                }
                if (!wait_or_abort(smem_addr(&dp_full), (uint32_t)(g & 1), limit, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                {
                    uint32_t raw[W];
                    tmem_ld_cols(lb + cPh, raw);
                    uint32_t pk[W / 2];
                    const uint64_t nd2 = f2_pack(-de, -de);
                    auto grads = [&](auto mask) {
                        constexpr bool M = decltype(mask)::value;
#pragma unroll
                        for (int x = 0; x < W / 2; ++x) {
                            const int c = 2 * x;
                            const uint64_t t = f2_add(f2_pack(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1])), nd2);
                            float d0, d1;
                            f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]), t), d0, d1);
                            if (M) {
                                d0 = p[c] != 0.f ? d0 : 0.f;
                                d1 = p[c + 1] != 0.f ? d1 : 0.f;
                            }
                            pk[x] = pack_bf16x2(d0, d1);
                        }
                    };
                    if (masked) grads(std::true_type{});
                    else grads(std::false_type{});
                    tmem_st_cols(lb + cPh, pk);  // dS over the dP columns already read
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_addr(&ds_ready));
            }
            if (!ok || !wait_or_abort(smem_addr(&o_full), (uint32_t)(it & 1), limit, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const size_t row = ((size_t)bh * N + qi) * prm.dreal;
#pragma unroll 1
            for (int c = hf; c < D / 32; c += E::NH) {  // this warp's 32-column chunks
                uint32_t raw[32];
                const int nc = min(32, prm.dreal - c * 32);
                tmem_ld32(lb + cQ + c * 32, raw);
                if (qi < N && nc > 0) store_row32(prm.dq, prm.g_fp32, row + c * 32, raw, prm.scale, nc);
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&acc_empty));  // dQ read: the next item may overwrite it
            if constexpr (!PERSIST) break;  // one item per CTA
            have = item(it + 1, q0, bh, n_steps);
        }
        if (!ok && !abort_flag) fail_bwd(&abort_flag);
    }
    // launched as a programmatic dependent of the dK/dV kernel: finish only
    // after it has, so that work after this kernel sees both
    pdl_wait_prior();
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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

template <int D, bool CAUSAL>
cudaError_t launch_dims(const BackwardProblem &p, float *delta, float *lse2, int pitch, cudaStream_t stream,
                        const char **detail)
{
    using C = BCfg<D>;
    const int64_t BH = p.B * p.H;
    CUtensorMap mq, mk, mv, mg;
    // maps of the real width: a padded head's missing columns load as zeros
    if (!make_map(&mq, p.q, BH, p.N, p.d) || !make_map(&mk, p.k, BH, p.N, p.d) || !make_map(&mv, p.v, BH, p.N, p.d) ||
        !make_map(&mg, p.dout, BH, p.N, p.d)) {
        *detail = "cuTensorMapEncodeTiled failed or is unavailable";
        return cudaErrorInvalidValue;
    }
    BwdParams prm;
    prm.N = (int)p.N;
    prm.BH = (int)BH;
    prm.n_q = (int)((p.N + BM - 1) / BM);
    {   // causal dQ order: as many heads per group as keep their K and V within half of L2
        int dev = 0, l2 = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            l2 = 0;
        const int64_t kv_head = p.N * p.d * 4;
        const int64_t g = l2 > 0 ? (int64_t)l2 / 2 / std::max<int64_t>(kv_head, 1) : BH;
        prm.hgroup = (int)std::max<int64_t>(1, std::min<int64_t>(g, BH));
    }
    prm.pitch = pitch;
    prm.dreal = (int)p.d;
    prm.sl = p.scale * 1.4426950408889634f;
    prm.scale = p.scale;
    prm.limit = 2000000000ull;
    prm.lse2 = lse2;
    prm.delta = delta;
    prm.dq = p.dq;
    prm.dk = p.dk;
    prm.dv = p.dv;
    prm.g_fp32 = p.grad_dtype == 1;
    // Short items (at most PERSIST_MAX_COLS streamed tiles x d: 16 tiles at
    // d = 128, 32 at d = 64) on persistent CTAs, one per SM, when there are more
    // of them than SMs: each item's prologue (resident loads, first score
    // products) and epilogue then overlap its neighbours' steps.  Longer items
    // run one per CTA (persistent, they measured -1 to -7 % at d = 128).
    cudaError_t e = cudaSuccess;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t items = (int64_t)prm.n_q * BH;
    const bool persist = prm.n_q * D <= PERSIST_MAX_COLS && items > sms;
    auto kv = persist ? fa_bwd_dkdv_tc<D, CAUSAL, true> : fa_bwd_dkdv_tc<D, CAUSAL, false>;
    auto kq = persist ? fa_bwd_dq_tc<D, CAUSAL, true> : fa_bwd_dq_tc<D, CAUSAL, false>;
    if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_KV_REQ)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_Q_REQ)) != cudaSuccess) return e;
    const unsigned grid = (unsigned)(persist ? std::min<int64_t>(items, sms) : items);
    kv<<<grid, EW<D>::NUM_THREADS, C::SMEM_KV_REQ, stream>>>(mq, mk, mv, mg, prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // programmatic dependent launch: the dQ CTAs (which read nothing the dK/dV
    // kernel writes) start on the SMs its last wave leaves idle
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(EW<D>::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_Q_REQ;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kq, mq, mk, mv, mg, prm);
}

}  // namespace

// bf16 heads of width 64 or 128, and narrower multiples of 8 padded up to them.
bool backward_tc_supported(const BackwardProblem &p)
{
    if (p.in_dtype != 0 || p.d < 8 || p.d > 128 || p.d % 8 != 0 || !(p.scale > 0.f)) return false;
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    return al16(p.q) && al16(p.k) && al16(p.v) && al16(p.dout) && al16(p.dq) && al16(p.dk) && al16(p.dv);
}

cudaError_t launch_backward_tc(const BackwardProblem &p, void *workspace, cudaStream_t stream, const char **detail)
{
    const int pitch = (int)((p.N + 127) / 128 * 128);
    float *delta = nullptr, *lse2 = nullptr;
    cudaError_t e = launch_backward_delta(p, workspace, stream, pitch, &delta, &lse2);
    if (e != cudaSuccess) return e;
    if (p.d > 64)
        return p.causal ? launch_dims<128, true>(p, delta, lse2, pitch, stream, detail)
                        : launch_dims<128, false>(p, delta, lse2, pitch, stream, detail);
    return p.causal ? launch_dims<64, true>(p, delta, lse2, pitch, stream, detail)
                    : launch_dims<64, false>(p, delta, lse2, pitch, stream, detail);
}

cudaError_t bwd_error_word_ptr(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_bwd_error_word);
}

}  // namespace fa
