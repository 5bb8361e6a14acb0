// Tensor-core attention forward for sm_103a: TMA -> shared memory ->
// tcgen05.mma into tensor memory, warp-specialised online softmax.
//
// Algorithm: the tiled online-softmax forward of "Deep Learning - Flash
// Attention" ("An Example", steps 4-7) and "FlashAttention" (ai360xpert.com,
// "Tiling and online softmax"), in the unnormalised form -- O and l are
// multiplied by alpha = 2^(m_old - m_new) when a key tile raises the running
// row maximum, P = 2^(S * scale * log2 e - m_new) feeds O += P V, and O is
// divided by l once after the last key tile.  Scores live in log2 units so
// each weight is one FFMA and one ex2.
//
// A work item is two 128-row query tiles (Q0, Q1) of one (batch, head); a CTA
// processes one item, or (short items) loops over items in rounds (item_index)
// with one CTA per SM.  Unmasked items of a head are adjacent; causal items
// run longest first within groups of heads whose K/V fit in half of L2
// (item_of).  A CTA streams the head's K/V tiles (128 keys) through a
// shared-memory ring:
//
//   warp 8  (TMA)      loads Q0, Q1 once per item (after the previous item's
//                      last S MMA) and stage j = (K_j, V_(j-1)) into the ring
//                      (one full/empty mbarrier pair per stage);
//   warp 9  (MMA)      allocates tensor memory and issues (one elected lane)
//                      S_t = Q_t K_j^T (SS form) and O_t += P_t V_j (A operand
//                      read from tensor memory), alternating the two tiles so
//                      the tensor core works on one tile while the other
//                      tile's softmax runs;
//   warps 0-3 / 4-7    softmax for Q0 / Q1: one query row per thread (a warp
//                      reads its 32 tensor-memory lanes), row max, weights,
//                      row sum, bf16 P written back over S, the alpha rescale
//                      of O in tensor memory, and the epilogue (O / l, LSE),
//                      which releases O_t (o_empty) as soon as it is read so
//                      the next item's first P V product can start.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [  0,128) S0 / P0   [128,256) S1 / P1   [256, 256+D) O0   [256+D, 256+2D) O1
// At D = 128, P_t (bf16, two per column) overwrites the first 64 columns of
// S_t; the next S_t MMA is issued after the P_t V MMA, and MMAs from one
// thread run in issue order.  At D = 64, P_t has columns of its own,
// [384 + 64 t, ...), so the next S_t MMA waits only for S_t to be read, and
// the MMAs are issued tile by tile (S_0(j+1), P_0 V, then S_1(j+1), P_1 V).
// At D = 128 the softmax warps release P_t in two halves (keys 0-63, then
// 64-127) and the P_t V product starts on the first; at D = 64 they release
// it whole, which saves the MMA warp a wait per tile.
//
// With a caller workspace and too few items to fill the GPU, items are
// further split over key ranges (SPLIT): each writes unnormalised O, m, l and
// the bf16 correction of its range, and a combine kernel merges them.
//
// Unmasked problems of at most 128 query rows, or with too few two-tile items
// to fill half of the SMs, run items of a single query tile (ONE): Q1's shared
// memory goes to a deeper K/V ring, the two softmax warpgroups take the even
// and the odd key tiles into the S0/P0/O0 and S1/P1/O1 slots, and warps 0-3
// merge the two partial results (m, l, O) before the epilogue.
//
// Every mbarrier wait is bounded (a caller-given limit in ns).  A wait that
// gives up sets the device error word and a CTA-wide abort flag; every role
// then leaves its loop, the MMA thread waits for its issued MMAs, the TMA
// thread for its issued loads, and tensor memory is freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace fa {

__device__ uint32_t g_tc_error_word;

namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = 128;           // query rows per tile (tensor-memory lanes)
constexpr int BN = 128;           // keys per tile
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int NUM_THREADS = 320;  // 10 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;  // lazy-rescale threshold, log2 units
constexpr int MAX_PARTS = 2;          // key slices P_t is released in, at most (Cfg::P_PARTS)

// error word bits
constexpr uint32_t ERR_WAIT_TMA = 1u;       // producer gave up waiting for a free slot
constexpr uint32_t ERR_WAIT_MMA = 2u;       // MMA thread gave up waiting for data or P
constexpr uint32_t ERR_WAIT_SOFTMAX = 4u;   // softmax gave up waiting for S or O
constexpr uint32_t ERR_DRAIN = 8u;          // teardown could not confirm in-flight work

constexpr int MAX_KVS = 6;            // key/value ring stages, at most

template <int DK, int DV, bool ONE = false>
struct Cfg {
    static constexpr int QCH = DK / 64;                    // 128-byte swizzle chunks of a Q/K row
    static constexpr int VCH = DV / 64;                    // ... of a V row
    static constexpr uint32_t Q_BYTES = BM * DK * 2;       // one 128 x DK bf16 tile
    static constexpr uint32_t K_BYTES = BN * DK * 2;
    static constexpr uint32_t V_BYTES = BN * DV * 2;
    static constexpr int Q_TILES = ONE ? 1 : 2;            // query tiles of an item
    // Ring of key/value stages: stage j holds K_j and V_(j-1), the two tiles
    // that iteration j of the MMA loop reads.  Two query tiles: three stages
    // when they fit in shared memory, else two.  One query tile (a short query
    // against a long key range: loading is most of the time): as many as fit
    // beside 2 KB of static shared memory, up to MAX_KVS, so each SM keeps more
    // bytes in flight (d = 128: 3, d = 64: 6).
    static constexpr int KVS_FIT = (int)((227u * 1024u - 1024u - 2048u - Q_BYTES) / (K_BYTES + V_BYTES));
    static constexpr int KVS = ONE ? (KVS_FIT < MAX_KVS ? KVS_FIT : MAX_KVS)
                                   : ((2 * Q_BYTES + 3 * (K_BYTES + V_BYTES) + 1024 <= 227u * 1024u) ? 3 : 2);
    static_assert(KVS >= 2 && KVS <= MAX_KVS, "key/value ring size");
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = Q_TILES * Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KVS * K_BYTES;
    static constexpr uint32_t SMEM_TILES = OFF_V + KVS * V_BYTES;
    static constexpr uint32_t SMEM_BYTES = SMEM_TILES + 1024;  // + alignment slack
    static constexpr uint32_t COL_O = 256;                 // O0 at 256, O1 at 256 + DV
    // DV = 64 leaves 128 tensor-memory columns free: P_t gets columns of its
    // own (64 packed columns each) instead of overwriting S_t, so S_t(j+1) can
    // be issued as soon as the softmax warps have read S_t(j)
    static constexpr bool SEP_P = DV == 64;
    static constexpr uint32_t COL_P = 256 + 2 * DV;        // P0 at COL_P, P1 at COL_P + 64 (SEP_P)
    // P_t is released to the P V product in this many key slices.  D = 128:
    // two halves (+3-5 % over one; four quarters measured 8 % slower than
    // halves).  D = 64: whole (+2.5 % on multi-head d = 64 over halves, every
    // wait the MMA warp saves counting among its many N = 64 products;
    // quarters -18 %).
    static constexpr int P_PARTS = DV == 64 ? 1 : 2;
};

struct Params {
    int N;             // query sequence length
    int Nk;            // key sequence length
    int H;             // heads
    int BH;            // batch * heads
    int n_qblocks;     // work items per head (256 query rows each; 128 for single-tile items)
    int n_items;       // n_qblocks * BH; see item_index for the CTA -> item order
    int hgroup;        // causal: heads per group of the item order (see item_of)
    int n_kv;          // key tiles per head
    float scale_log2;  // scale * log2(e), > 0
    int causal;
    int skip_load;     // fault injection: never issue the K load of this tile (-1 = off)
    uint64_t wait_limit_ns;
    void *o;
    int64_t os_b, os_h, os_n;  // O element strides (batch, head, sequence)
    int qperm, kperm, vperm;   // which of (sequence, head, batch) each outer map dimension holds
    float *lse;
    int o_fp32;
    int dv_real;       // O columns stored (<= DV: narrower heads are padded with zeros)
    // key-range split (n_split > 1): each item covers key tiles [kv_per sp, kv_per (sp + 1))
    // and writes unnormalised partials instead of O and LSE
    int n_split, kv_per;
    float *o_part, *m_part, *l_part, *d_part;
};

struct __align__(8) Barriers {
    uint64_t q_full[2], q_empty;      // query tiles of an item; free after its last S MMA
    uint64_t kv_full[MAX_KVS], kv_empty[MAX_KVS];
    uint64_t s_full[2];
    uint64_t p_part[2][MAX_PARTS];    // P_t keys [0, (k + 1) BN / P_PARTS) written
    uint64_t s_read[2], p_free[2];    // SEP_P: S_t read by the softmax warps / P_t read by the P V product
    uint64_t o_full[2], o_empty[2];   // O_t complete / read by the epilogue
    uint64_t part_full, part_empty;   // single-tile items: the odd key tiles' m, l, dq written / read
    uint64_t drain;
};

// A work item: two 128-row query tiles (256 rows) of one (batch, head).
struct Item {
    int bh, b, h;
    int qrow0;   // first row of Q0; Q1 starts BM later
    int n0, n1;  // key tiles each query tile needs: all, or up to its diagonal under the mask
    int kv_lo;   // first key tile (key-range split; 0 otherwise)
    int sp;      // split index
};

// Item of this CTA's round `it`: rounds alternate direction over the CTAs
// (c, then G - 1 - c, ...), so with items sorted longest first (causal) every
// CTA's total stays close to the mean.  Increasing in `it`.
// Without persistence a CTA takes the single item blockIdx.x.
template <bool PERSIST>
__device__ __forceinline__ int item_index(int it)
{
    if (!PERSIST) return it == 0 ? (int)blockIdx.x : INT_MAX;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    return it * G + ((it & 1) ? G - 1 - c : c);
}

template <bool CAUSAL, bool SPLIT, bool ONE>
__device__ __forceinline__ Item item_of(const Params &prm, int w)
{
    int qb, bh, sp = 0;
    if (SPLIT) {
        sp = w % prm.n_split;
        w /= prm.n_split;
    }
    if (CAUSAL) {
        // Heads in groups of hgroup whose keys and values fit in L2 together,
        // one group after the other; within a group the longest query blocks
        // first (the CTAs of short blocks fill in behind the long ones)
        const int per = prm.hgroup * prm.n_qblocks;
        const int g0 = (w / per) * prm.hgroup, x = w % per;
        const int gh = min(prm.hgroup, prm.BH - g0);  // heads in this group
        qb = prm.n_qblocks - 1 - x / gh;
        bh = g0 + x % gh;
    } else {       // items of one head are adjacent: concurrent CTAs share its K/V in L2
        qb = w % prm.n_qblocks;
        bh = w / prm.n_qblocks;
    }
    Item it;
    it.sp = sp;
    it.kv_lo = SPLIT ? sp * prm.kv_per : 0;
    it.bh = bh;
    it.b = bh / prm.H;
    it.h = bh % prm.H;
    it.qrow0 = qb * (ONE ? 1 : 2) * BM;
    it.n0 = CAUSAL ? min(prm.n_kv, 2 * qb + 1) : (SPLIT ? min(prm.n_kv - it.kv_lo, prm.kv_per) : prm.n_kv);
    it.n1 = CAUSAL ? min(prm.n_kv, 2 * qb + 2) : it.n0;
    return it;
}

// Map coordinate for dimension slot s of a tensor map whose outer dimensions
// are ordered by stride: 0 = sequence row, 1 = head, 2 = batch.
__device__ __forceinline__ int pick(int s, int row, int h, int b) { return s == 0 ? row : (s == 1 ? h : b); }

__device__ __forceinline__ void tma_load_rows(uint32_t dst, const void *tmap, uint32_t bar, int col, int perm, int row,
                                              int h, int b, uint64_t pol)
{
    tma_load_4d(dst, tmap, bar, col, pick(perm & 3, row, h, b), pick((perm >> 2) & 3, row, h, b),
                pick((perm >> 4) & 3, row, h, b), pol);
}

__device__ __forceinline__ void raise_error(uint32_t bit, volatile int *abort_flag)
{
    atomicOr(&g_tc_error_word, bit);
    *abort_flag = 1;
}

// Columns col0 .. col0 + ncols - 1 of an O row (ncols <= 32, a multiple of 8:
// a head dimension padded up to the kernel's stores only its own columns).
__device__ __forceinline__ void store_o_row(void *o, int o_fp32, size_t row_elem, const float *vals,
                                            int col0, int ncols)
{
    if (o_fp32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(o) + row_elem + col0);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            if (4 * x < ncols) dst[x] = make_float4(vals[4 * x], vals[4 * x + 1], vals[4 * x + 2], vals[4 * x + 3]);
        }
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o) + row_elem + col0);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            if (8 * x >= ncols) break;
            uint4 w;
            w.x = pack_bf16x2(vals[8 * x + 0], vals[8 * x + 1]);
            w.y = pack_bf16x2(vals[8 * x + 2], vals[8 * x + 3]);
            w.z = pack_bf16x2(vals[8 * x + 4], vals[8 * x + 5]);
            w.w = pack_bf16x2(vals[8 * x + 6], vals[8 * x + 7]);
            dst[x] = w;
        }
    }
}

// ONE: every item has a single query tile (unmasked problems of at most 128
// query rows per head, or with too few two-tile items to fill half of the
// SMs; see one_tile_items).  The two softmax warpgroups then share that tile's key tiles,
// even ones to warps 0-3 and odd ones to warps 4-7, each with its own running
// maximum, sum and O accumulator in the tile slots of S, P and O; warps 0-3
// merge the two partial results by the log-sum-exp rule before the epilogue.
template <int DK, int DV, bool CAUSAL, bool PERSIST, bool SPLIT, bool ONE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
fa_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const Params prm)
{
    using C = Cfg<DK, DV, ONE>;
    constexpr int P_PARTS = C::P_PARTS;
    static_assert(P_PARTS <= MAX_PARTS && (BN / 32) % P_PARTS == 0, "P slices must be whole 32-key chunks");
    extern __shared__ uint8_t smem_raw[];
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;
    __shared__ float part_mld[ONE ? 3 : 1][ONE ? BM : 1];  // ONE: m, l, dq of the odd key tiles, per row

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = prm.N, Nk = prm.Nk;

    // ---- setup (once per CTA; the CTA then loops over work items)
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_addr(&bars.q_full[t]), 1);
            mbar_init(smem_addr(&bars.s_full[t]), 1);
            for (int k = 0; k < P_PARTS; ++k) mbar_init(smem_addr(&bars.p_part[t][k]), 128);
            mbar_init(smem_addr(&bars.s_read[t]), 128);
            mbar_init(smem_addr(&bars.p_free[t]), 1);
            mbar_init(smem_addr(&bars.o_full[t]), 1);
            mbar_init(smem_addr(&bars.o_empty[t]), 128);
        }
        mbar_init(smem_addr(&bars.q_empty), 1);
        mbar_init(smem_addr(&bars.part_full), 128);
        mbar_init(smem_addr(&bars.part_empty), 128);
        for (int s = 0; s < C::KVS; ++s) {
            mbar_init(smem_addr(&bars.kv_full[s]), 1);
            mbar_init(smem_addr(&bars.kv_empty[s]), 1);
        }
        mbar_init(smem_addr(&bars.drain), 1);
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
    // The merge of the key-range partials may be scheduled now (it waits for this
    // grid to finish before reading); a split grid never has more CTAs than SMs,
    // so its blocks take only SMs this grid leaves idle.
    if constexpr (SPLIT) pdl_launch_dependents();

    if (warp == TMA_WARP) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_q = policy_evict_first();
            // K/V: kept in L2 for the other query blocks of the head, or, with a
            // single query block per head, read once
            const uint64_t pol_kv = prm.n_qblocks > 1 ? policy_evict_last() : policy_evict_first();
            int g = 0;                     // stages issued over all items (ring position)
            int q_items = 0;               // items whose Q loads were issued
            int skipped = -1;              // ring position of the injected, never-filled stage
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int w = item_index<PERSIST>(it);
                if (w >= prm.n_items) break;
                const Item wi = item_of<CAUSAL, SPLIT, ONE>(prm, w);
                // stage s of the item = K_s (s < n1) and V_(s-1) (s >= 1), s = 0 .. n1
                auto load_stage = [&](int s) -> bool {
                    const int slot = g % C::KVS;
                    const uint32_t n_use = (uint32_t)(g / C::KVS);
                    const uint32_t full = smem_addr(&bars.kv_full[slot]);
                    if (!wait_or_abort(smem_addr(&bars.kv_empty[slot]), (n_use & 1u) ^ 1u, limit, &abort_flag)) return false;
                    ++g;
                    if (it == 0 && s == prm.skip_load && s < wi.n1) {  // fault injection: this stage never fills
                        skipped = g - 1;
                        return true;
                    }
                    const bool has_k = s < wi.n1, has_v = s >= 1;
                    mbar_arrive_expect_tx(full, (has_k ? C::K_BYTES : 0u) + (has_v ? C::V_BYTES : 0u));
                    if (has_k)
                        for (int c = 0; c < C::QCH; ++c)
                            tma_load_rows(s_base + C::OFF_K + slot * C::K_BYTES + c * (BN * 128), &tm_k, full, c * 64,
                                          prm.kperm, (wi.kv_lo + s) * BN, wi.h, wi.b, pol_kv);
                    if (has_v)
                        for (int c = 0; c < C::VCH; ++c)
                            tma_load_rows(s_base + C::OFF_V + slot * C::V_BYTES + c * (BN * 128), &tm_v, full, c * 64,
                                          prm.vperm, (wi.kv_lo + s - 1) * BN, wi.h, wi.b, pol_kv);
                    return true;
                };
                // the first key tile may load before the previous item's last S MMA
                // frees the query tiles
                ok = load_stage(0);
                if (ok && it > 0 && !wait_or_abort(smem_addr(&bars.q_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag))
                    ok = false;
                if (ok) {
                    for (int t = 0; t < (ONE ? 1 : 2); ++t) {
                        const uint32_t bar = smem_addr(&bars.q_full[t]);
                        mbar_arrive_expect_tx(bar, C::Q_BYTES);
                        for (int c = 0; c < C::QCH; ++c)
                            tma_load_rows(s_base + C::OFF_Q + t * C::Q_BYTES + c * (BM * 128), &tm_q, bar, c * 64,
                                          prm.qperm, wi.qrow0 + t * BM, wi.h, wi.b, pol_q);
                    }
                    q_items = it + 1;
                }
                for (int s = 1; ok && s <= wi.n1; ++s) ok = load_stage(s);
            }
            if (!ok) {
                if (!abort_flag) raise_error(ERR_WAIT_TMA, &abort_flag);
            }
            // Before the CTA exits, every load issued must have landed.
            if (abort_flag) {
                for (int p = max(0, g - C::KVS); p < g; ++p) {
                    if (p == skipped) continue;
                    const uint32_t full = smem_addr(&bars.kv_full[p % C::KVS]);
                    if (!mbar_wait_bounded(full, (uint32_t)((p / C::KVS) & 1), limit)) atomicOr(&g_tc_error_word, ERR_DRAIN);
                }
                if (q_items > 0)
                    for (int t = 0; t < (ONE ? 1 : 2); ++t)
                        if (!mbar_wait_bounded(smem_addr(&bars.q_full[t]), (uint32_t)((q_items - 1) & 1), limit))
                            atomicOr(&g_tc_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================================================================ MMA issuer
        // The whole warp runs this branch converged; elect.sync picks the lane
        // that issues each MMA and commit.
        {
            const uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(BM, DV, 0, 1);
            const uint32_t sQ = s_base + C::OFF_Q, sK = s_base + C::OFF_K, sV = s_base + C::OFF_V;
            bool ok = true;
            bool issued_any = false;
            auto wait = [&](uint64_t *b, uint32_t parity) -> bool {
                if (!ok) return false;
                const bool done = wait_or_abort(smem_addr(b), parity, limit, &abort_flag);
                if (!__all_sync(0xffffffffu, done)) {  // reconverges the warp; one outcome for all lanes
                    ok = false;
                    if (!abort_flag) raise_error(ERR_WAIT_MMA, &abort_flag);
                    return false;
                }
                return true;
            };
            // Descriptors are built once; a K step only moves the start address
            // (field bits 0-13 hold address >> 4, and every shared-memory
            // address here is below 256 KB, so adding offset >> 4 never carries
            // out of the field).
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024), dq1 = sdesc_sw128(sQ + C::Q_BYTES, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sK, 16, 1024), dv0 = sdesc_sw128(sV, BN * 128, 1024);
            constexpr uint64_t K_STEP = C::K_BYTES >> 4, V_STEP = C::V_BYTES >> 4;  // one ring slot, descriptor units
            // S_t = Q_t K^T from ring slot `slot` (M = 128 rows, N = 128 keys, K = D in steps of 16)
            auto mma_s = [&](int t, int slot) {
                const uint64_t q = (t && !ONE) ? dq1 : dq0, k = dk0 + (uint64_t)slot * K_STEP;
                const uint32_t d_s = tmem + t * 128;
                uint64_t qa[DK / 16], kb[DK / 16];
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4);
                    qa[kk] = q + off;
                    kb[kk] = k + off;
                }
                mma_ss_k<DK / 16>(d_s, qa, kb, idesc_s, 0u);  // the K loop under one election
                issued_any = true;
            };
            // O_t += P_t V from ring slot `slot` (M = 128 rows, N = D, K = 128 keys in steps of 16);
            // `first` starts the accumulator (key tile 0)
            // slice `h` of the keys (BN / P_PARTS of them): a slice starts while the
            // softmax warps still compute the later ones
            auto mma_o = [&](int t, int slot, bool first, int h) {
                const uint64_t v = dv0 + (uint64_t)slot * V_STEP;
                const uint32_t d_o = tmem + C::COL_O + t * DV, a_p = tmem + (C::SEP_P ? C::COL_P + t * 64 : t * 128);
                constexpr int KS = BN / 16 / P_PARTS;  // K steps per slice
                uint32_t pa[KS];
                uint64_t vb[KS];
#pragma unroll
                for (int x = 0; x < KS; ++x) {
                    const int kk = KS * h + x;
                    pa[x] = a_p + kk * 8;
                    vb[x] = v + (uint64_t)((kk * 16 * 128) >> 4);
                }
                mma_ts_k<KS>(d_o, pa, vb, idesc_o, (!first || h > 0) ? 1u : 0u);
                issued_any = true;
            };
            int slot = 0;            // ring slot of the current stage
            uint32_t phase = 0;      // its fill parity
            auto next_stage = [&]() {
                if (++slot == C::KVS) {
                    slot = 0;
                    phase ^= 1u;
                }
            };
            uint32_t pp[2] = {0u, 0u};  // P releases waited for so far, per tile
            uint32_t ns[2] = {0u, 0u};  // S_t products issued so far (SEP_P)
            for (int it = 0; ok; ++it) {
                const int w = item_index<PERSIST>(it);
                if (w >= prm.n_items) break;
                const Item wi = item_of<CAUSAL, SPLIT, ONE>(prm, w);
                const int n0 = wi.n0, n1 = wi.n1;
                // the first P_t V product of an item overwrites O_t: the previous
                // item's epilogue must have read it
                auto o_free = [&](int t) -> bool { return it == 0 || wait(&bars.o_empty[t], (uint32_t)((it - 1) & 1)); };
                // O_t += P_t V slice by slice, each once its slice of P_t is written
                auto pv = [&](int t, int slot, bool first) -> bool {
                    const uint32_t par = pp[t] & 1u;
                    ++pp[t];
#pragma unroll
                    for (int h = 0; h < P_PARTS; ++h) {
                        if (!wait(&bars.p_part[t][h], par) || (h == 0 && first && !o_free(t))) return false;
                        tc_fence_after();
                        mma_o(t, slot, first, h);
                    }
                    return true;
                };
                // Before S_t is overwritten the softmax warps must have read the
                // previous S_t (ns[t] S_t products so far over all items).
                auto s_free = [&](int t) -> bool {
                    const bool r = ns[t] == 0 || wait(&bars.s_read[t], (ns[t] - 1) & 1u);
                    ++ns[t];
                    return r;
                };
                if constexpr (ONE && C::SEP_P) {
                    // Key tile k goes to slot k mod 2.  P has columns of its own, so
                    // S(k + 2) is issued as soon as the slot's softmax warps have read
                    // S(k), ahead of P(k) V: they find their next scores ready when they
                    // finish a tile.  Two ring positions: `ws` is the next stage to wait
                    // for (its K feeds an S product), `slot` the next to release (its V
                    // feeds P V); stage j is released after P(j - 1) V, stage 0 after S(0).
                    int ws = slot;
                    uint32_t wph = phase;
                    auto next_w = [&]() {
                        if (++ws == C::KVS) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    };
                    auto s_at = [&](int t) -> bool {  // S_t = Q K from stage ws
                        if (!s_free(t)) return false;
                        tc_fence_after();
                        mma_s(t, ws);
                        mma_commit_w(smem_addr(&bars.s_full[t]));
                        return true;
                    };
                    auto pv_stage = [&](int u, bool first, bool last) -> bool {
                        if (!pv(u, slot, first)) return false;
                        mma_commit_w(smem_addr(&bars.p_free[u]));
                        if (last) mma_commit_w(smem_addr(&bars.o_full[u]));
                        return true;
                    };
                    if (!wait(&bars.q_full[0], (uint32_t)(it & 1))) break;
                    for (int k = 0; ok && k < 2 && k < n0; ++k) {
                        if (!wait(&bars.kv_full[ws], wph) || !(k ? s_at(1) : s_at(0))) break;
                        if (PERSIST && k == n0 - 1) mma_commit_w(smem_addr(&bars.q_empty));
                        next_w();
                    }
                    if (!ok) break;
                    mma_commit_w(smem_addr(&bars.kv_empty[slot]));  // stage 0: K_0 only
                    next_stage();
                    for (int k = 0; ok && k < n0; ++k) {
                        if (k + 2 < n0) {
                            if (!wait(&bars.kv_full[ws], wph) || !((k & 1) ? s_at(1) : s_at(0))) break;
                            if (PERSIST && k + 2 == n0 - 1) mma_commit_w(smem_addr(&bars.q_empty));
                            next_w();
                        }
                        // stage k + 1 (K_(k+1), V_k) was waited for when S(k + 1) was
                        // issued; the last stage holds V only
                        if (k + 1 == n0 && !wait(&bars.kv_full[slot], phase)) break;
                        const bool first = k < 2, last = k + 2 >= n0;  // slot's first / last key tile
                        if (!((k & 1) ? pv_stage(1, first, last) : pv_stage(0, first, last))) break;
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                        next_stage();
                    }
                } else if constexpr (ONE) {
                    // Stage s holds K_s and V_(s-1).  Key tile s goes to slot t = s mod 2
                    // (S_t = Q K_s), and P_u V_(s-1) for u = 1 - t completes key tile
                    // s - 1.  S_t is issued first: slot t's previous P_t V product was
                    // issued a stage earlier, so it is ordered before the overwrite.
                    // (the tile slot t or u is passed as a literal at each call, so the
                    // per-tile counters pp[] and ns[] stay in registers)
                    auto s_stage = [&](int t) -> bool {
                        if (C::SEP_P && !s_free(t)) return false;
                        tc_fence_after();
                        mma_s(t, slot);
                        mma_commit_w(smem_addr(&bars.s_full[t]));
                        return true;
                    };
                    auto pv_stage = [&](int u, bool first, bool last) -> bool {
                        if (!pv(u, slot, first)) return false;
                        if (C::SEP_P) mma_commit_w(smem_addr(&bars.p_free[u]));
                        if (last) mma_commit_w(smem_addr(&bars.o_full[u]));
                        return true;
                    };
                    for (int s = 0; ok && s <= n0; ++s) {
                        if (!wait(&bars.kv_full[slot], phase)) break;
                        if (s == 0 && !wait(&bars.q_full[0], (uint32_t)(it & 1))) break;
                        if (s < n0) {
                            if (!((s & 1) ? s_stage(1) : s_stage(0))) break;
                            if (PERSIST && s == n0 - 1) mma_commit_w(smem_addr(&bars.q_empty));
                        }
                        if (s >= 1) {
                            // key tiles 0 and 1 start O_0 and O_1; slot u's last key tile is s - 1
                            // when no key tile s + 1 follows
                            const bool first = s - 1 < 2, last = s + 1 >= n0;
                            if (!((s & 1) ? pv_stage(0, first, last) : pv_stage(1, first, last))) break;
                        }
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                        next_stage();
                    }
                } else if constexpr (C::SEP_P) {
                    // stage 0: K_0
                    if (wait(&bars.q_full[0], (uint32_t)(it & 1)) && wait(&bars.kv_full[slot], phase) && s_free(0)) {
                        tc_fence_after();
                        mma_s(0, slot);
                        mma_commit_w(smem_addr(&bars.s_full[0]));
                    }
                    if (wait(&bars.q_full[1], (uint32_t)(it & 1)) && s_free(1)) {
                        tc_fence_after();
                        mma_s(1, slot);
                        mma_commit_w(smem_addr(&bars.s_full[1]));
                        if (PERSIST && n1 == 1) mma_commit_w(smem_addr(&bars.q_empty));
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                    }
                    next_stage();
                    // iteration j reads stage j + 1 (K_(j+1), V_j), tile by tile: S_t(j+1)
                    // as soon as S_t(j) is read, then P_t(j) V_j.  Tile 0's products go
                    // first, so they never wait behind tile 1's softmax.
                    for (int j = 0; ok && j < n1; ++j) {
                        if (!wait(&bars.kv_full[slot], phase)) break;
                        if (j + 1 < n0) {
                            if (!s_free(0)) break;
                            tc_fence_after();
                            mma_s(0, slot);
                            mma_commit_w(smem_addr(&bars.s_full[0]));
                        }
                        if (j < n0) {
                            if (!pv(0, slot, j == 0)) break;
                            mma_commit_w(smem_addr(&bars.p_free[0]));
                            if (j == n0 - 1) mma_commit_w(smem_addr(&bars.o_full[0]));
                        }
                        if (j + 1 < n1) {
                            if (!s_free(1)) break;
                            tc_fence_after();
                            mma_s(1, slot);
                            mma_commit_w(smem_addr(&bars.s_full[1]));
                            if (PERSIST && j + 1 == n1 - 1) mma_commit_w(smem_addr(&bars.q_empty));
                        }
                        if (!pv(1, slot, j == 0)) break;
                        mma_commit_w(smem_addr(&bars.p_free[1]));
                        if (j == n1 - 1) mma_commit_w(smem_addr(&bars.o_full[1]));
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                        next_stage();
                    }
                } else {
                    // stage 0: K_0
                    if (wait(&bars.q_full[0], (uint32_t)(it & 1)) && wait(&bars.kv_full[slot], phase)) {
                        tc_fence_after();
                        mma_s(0, slot);
                        mma_commit_w(smem_addr(&bars.s_full[0]));
                    }
                    if (wait(&bars.q_full[1], (uint32_t)(it & 1))) {
                        tc_fence_after();
                        mma_s(1, slot);
                        mma_commit_w(smem_addr(&bars.s_full[1]));
                        if (PERSIST && n1 == 1) mma_commit_w(smem_addr(&bars.q_empty));
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                    }
                    next_stage();
                    // iteration j reads stage j (K_j, V_(j-1)): P_t V_(j-1), then S_t = Q_t K_j^T
                    for (int j = 1; ok && j < n1; ++j) {
                        if (!wait(&bars.kv_full[slot], phase)) break;
                        // tile 0
                        if (j <= n0) {
                            if (!pv(0, slot, j == 1)) break;
                            if (j < n0) {
                                mma_s(0, slot);
                                mma_commit_w(smem_addr(&bars.s_full[0]));
                            } else {
                                mma_commit_w(smem_addr(&bars.o_full[0]));
                            }
                        }
                        // tile 1
                        if (!pv(1, slot, j == 1)) break;
                        mma_s(1, slot);
                        mma_commit_w(smem_addr(&bars.s_full[1]));
                        if (PERSIST && j == n1 - 1) mma_commit_w(smem_addr(&bars.q_empty));  // the item's last S MMA
                        mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                        next_stage();
                    }
                    if (!ok) break;
                    // stage n1: V of the last key tile
                    const int last = n1 - 1;
                    if (!wait(&bars.kv_full[slot], phase)) break;
                    if (n0 == n1) {
                        if (!pv(0, slot, last == 0)) break;
                        mma_commit_w(smem_addr(&bars.o_full[0]));
                    }
                    if (!pv(1, slot, last == 0)) break;
                    mma_commit_w(smem_addr(&bars.o_full[1]));
                    mma_commit_w(smem_addr(&bars.kv_empty[slot]));
                    next_stage();
                }
            }
            if (!ok && issued_any) {
                // every MMA issued so far must finish before tensor memory is freed
                mma_commit_w(smem_addr(&bars.drain));
                if (!mbar_wait_bounded(smem_addr(&bars.drain), 0, limit) && lane == 0)
                    atomicOr(&g_tc_error_word, ERR_DRAIN);
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax + epilogue
        const int t = warp >> 2;          // query tile 0 or 1
        const int quarter = warp & 3;     // tensor-memory lanes 32*quarter ...
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tS = lane_base + t * 128;
        const uint32_t tO = lane_base + C::COL_O + t * DV;
        const uint32_t tP = C::SEP_P ? lane_base + C::COL_P + t * 64 : tS;  // where P_t goes
        const float sl = prm.scale_log2;
        uint32_t sp = 0;                  // s_full waits so far
        uint32_t np = 0;                  // P_t tiles written so far (SEP_P: p_free phases)
        bool ok = true;
        auto fail = [&]() {
            ok = false;
            if (!abort_flag) raise_error(ERR_WAIT_SOFTMAX, &abort_flag);
            else atomicOr(&g_tc_error_word, ERR_WAIT_SOFTMAX);
        };
        for (int it = 0; ok; ++it) {
            const int w = item_index<PERSIST>(it);
            if (w >= prm.n_items) break;
            const Item wi = item_of<CAUSAL, SPLIT, ONE>(prm, w);
            const int grow = wi.qrow0 + (ONE ? 0 : t * BM) + r;  // global query row of this thread
            // key tiles of this warpgroup (ONE: every other one, from key tile t)
            const int n_t = ONE ? (wi.n0 + 1 - t) >> 1 : (t == 0 ? wi.n0 : wi.n1);
            // every row of this warp is padding (short or ragged queries): the warp
            // keeps its place in the barrier sequence -- the waits order its
            // arrivals after the others' of the same tile -- but skips the scores,
            // the weights and their tensor-memory traffic.  Its O rows are never stored.
            const bool idle = grow - lane >= N;
            float m = -INFINITY;  // running maximum, log2 units
            float l = 0.f;        // running denominator (exact weights): LSE
            float dq = 0.f;       // bf16 rounding of each tile's largest weight: O / (l + dq)
            for (int j = 0; j < n_t; ++j) {
                if (!wait_or_abort(smem_addr(&bars.s_full[t]), sp & 1u, limit, &abort_flag)) {
                    fail();
                    break;
                }
                ++sp;
                if (idle) {
                    if constexpr (C::SEP_P) mbar_arrive(smem_addr(&bars.s_read[t]));
                    if (C::SEP_P && np > 0 && !wait_or_abort(smem_addr(&bars.p_free[t]), (np - 1) & 1u, limit, &abort_flag)) {
                        fail();
                        break;
                    }
                    ++np;
#pragma unroll
                    for (int h = 0; h < P_PARTS; ++h) mbar_arrive(smem_addr(&bars.p_part[t][h]));
                    continue;
                }
                tc_fence_after();
                float s[BN];
                {
                    uint32_t raw[BN];
                    tmem_ld128(tS, raw);
#pragma unroll
                    for (int x = 0; x < BN; ++x) s[x] = __uint_as_float(raw[x]);
                }
                if constexpr (C::SEP_P) {  // S_t is in registers: the next S_t product may start
                    tc_fence_before();
                    mbar_arrive(smem_addr(&bars.s_read[t]));
                }
                const int kv0 = (wi.kv_lo + (ONE ? 2 * j + t : j)) * BN;
                int lim = Nk - kv0;                         // keys >= Nk are padding
                if (CAUSAL) lim = min(lim, grow - kv0 + 1);  // keys after this query
                if (lim < BN) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                const float mx = row_max<BN>(s);
                const float m_tile = mx * sl;
                // Lazy rescaling: the reference maximum m moves only when the tile's
                // maximum exceeds it by more than RESCALE_LOG2 (weights then stay
                // below 2^RESCALE_LOG2).  Softmax is invariant to the shift, so O / l
                // and m + log2 l are unchanged; alpha is 1 on most tiles.
                float alpha = 1.f;
                if (m_tile > m + RESCALE_LOG2) {
                    alpha = ex2(m - m_tile);  // 0 on the first tile (m = -inf)
                    m = m_tile;
                }
                // O_t already holds every earlier P V product of this item (the
                // commit that signalled this S tile covers all MMAs issued before
                // it; with P_t in columns of its own, the wait for the previous
                // P_t's product to finish reading them covers it); rescale it
                // before any P V product of this tile is released.
                if (C::SEP_P && np > 0 && !wait_or_abort(smem_addr(&bars.p_free[t]), (np - 1) & 1u, limit, &abort_flag)) {
                    fail();
                    break;
                }
                ++np;
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                    for (int c = 0; c < DV / 16; ++c) {  // 16 columns at a time: the scores are live
                        uint32_t raw[16];
                        tmem_ld16(tO + c * 16, raw);
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            float o0, o1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(raw[2 * x]), __uint_as_float(raw[2 * x + 1])), a2), o0, o1);
                            raw[2 * x] = __float_as_uint(o0);
                            raw[2 * x + 1] = __float_as_uint(o1);
                        }
                        tmem_st16(tO + c * 16, raw);
                    }
                }
                const float base = (m == -INFINITY) ? 0.f : m;  // a row with no key yet
                const uint64_t sl2 = f2_pack(sl, sl), nb2 = f2_pack(-base, -base);
                uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        float a0, a1;
                        f2_unpack(f2_fma(f2_pack(s[c * 32 + 2 * x], s[c * 32 + 2 * x + 1]), sl2, nb2), a0, a1);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        pk[x] = pack_bf16x2(p0, p1);
                        rs2[x & 1] = f2_add(rs2[x & 1], f2_pack(p0, p1));
                    }
                    tmem_st16(tP + c * 16, pk);
                    constexpr int CPP = BN / 32 / P_PARTS;  // 32-key chunks per slice
                    if ((c + 1) % CPP == 0 && c + 1 < BN / 32) {  // a slice of P is written: its P V may start
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(smem_addr(&bars.p_part[t][c / CPP]));
                    }
                }
                float r0, r1;
                f2_unpack(f2_add(rs2[0], rs2[1]), r0, r1);
                l = l * alpha + (r0 + r1);
                // The P V product sees bf16 weights.  The largest weight of the
                // tile dominates a peaked row, so the normaliser of O gets that
                // weight's rounding error added: O's numerator and denominator then
                // agree on the terms that matter (the same FFMA and ex2 as above,
                // so p_top is bit-identical to that element's weight).
                const float p_top = ex2(fmaf(mx, sl, -base));
                dq = dq * alpha + (__uint_as_float(pack_bf16x2(p_top, 0.f) << 16) - p_top);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_addr(&bars.p_part[t][P_PARTS - 1]));
            }
            if (!ok) break;
            // ONE: warps 4-7 hand their rows' m, l, dq to warps 0-3 and are done
            // with the item; warps 0-3 merge O_1 into O_0 as they read it.  (Every
            // item of a persistent grid has the same key tiles, so the barriers
            // below change phase once per item, or never when there is one key tile.)
            if (ONE && t == 1) {
                if (n_t == 0) continue;
                if (it > 0 && !wait_or_abort(smem_addr(&bars.part_empty), (uint32_t)((it - 1) & 1), limit, &abort_flag)) {
                    fail();
                    break;
                }
                part_mld[0][r] = m;
                part_mld[1][r] = l;
                part_mld[2][r] = dq;
                mbar_arrive(smem_addr(&bars.part_full));
                continue;
            }
            // ---- epilogue: O / l, LSE.  O_t is read whole, then released to the
            // next item's first P V product before the stores.
            if (!wait_or_abort(smem_addr(&bars.o_full[t]), (uint32_t)(it & 1), limit, &abort_flag)) {
                fail();
                break;
            }
            tc_fence_after();
            const bool has1 = ONE && wi.n0 >= 2;  // ONE: O_1 holds the odd key tiles
            float w0 = 1.f, w1 = 0.f;             // their weights in the merged O
            if (has1) {
                if (!wait_or_abort(smem_addr(&bars.part_full), (uint32_t)(it & 1), limit, &abort_flag) ||
                    !wait_or_abort(smem_addr(&bars.o_full[1]), (uint32_t)(it & 1), limit, &abort_flag)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const float m1 = part_mld[0][r], l1 = part_mld[1][r], d1 = part_mld[2][r];
                mbar_arrive(smem_addr(&bars.part_empty));
                // the log-sum-exp merge of two key ranges: both sums and O move to
                // the larger reference maximum
                const float mm = fmaxf(m, m1);
                w0 = m == -INFINITY ? 0.f : ex2(m - mm);
                w1 = m1 == -INFINITY ? 0.f : ex2(m1 - mm);
                m = mm;
                l = w0 * l + w1 * l1;
                dq = w0 * dq + w1 * d1;
            }
            // 32 columns of O from column c * 32: O_t, or under ONE w0 O_0 + w1 O_1
            auto load_o = [&](int c, uint32_t (&raw)[32]) {
                tmem_ld32(tO + c * 32, raw);
                if (ONE && has1) {
                    uint32_t raw1[32];
                    tmem_ld32(tO + DV + c * 32, raw1);
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        raw[x] = __float_as_uint(fmaf(w0, __uint_as_float(raw[x]), w1 * __uint_as_float(raw1[x])));
                }
            };
            // releases the O columns this epilogue read (persistent grids)
            auto release_o = [&]() {
                tc_fence_before();
                mbar_arrive(smem_addr(&bars.o_empty[t]));
                if (has1) mbar_arrive(smem_addr(&bars.o_empty[1]));
            };
            if constexpr (SPLIT) {  // key-range partials: unnormalised O, m, l, dq
                const size_t prow = ((size_t)wi.sp * prm.BH + wi.bh) * N + grow;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t raw[32];
                    load_o(c, raw);
                    if (grow < N) {
                        float4 *dst = reinterpret_cast<float4 *>(prm.o_part + prow * DV + c * 32);
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            dst[x] = make_float4(__uint_as_float(raw[4 * x]), __uint_as_float(raw[4 * x + 1]),
                                                 __uint_as_float(raw[4 * x + 2]), __uint_as_float(raw[4 * x + 3]));
                    }
                }
                if (PERSIST) release_o();
                if (grow < N) {
                    prm.m_part[prow] = m;
                    prm.l_part[prow] = l;
                    prm.d_part[prow] = dq;
                }
                continue;
            }
            const float inv_l = 1.f / (l + dq);
            const size_t row_elem = (size_t)(wi.b * prm.os_b + wi.h * prm.os_h + (int64_t)grow * prm.os_n);
            if (PERSIST && !ONE) {
                uint32_t ov[DV];
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(tO + c * 32, raw);
#pragma unroll
                    for (int x = 0; x < 32; ++x) ov[c * 32 + x] = raw[x];
                }
                tc_fence_before();
                mbar_arrive(smem_addr(&bars.o_empty[t]));
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    float vals[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) vals[x] = __uint_as_float(ov[c * 32 + x]) * inv_l;
                    const int nc = min(32, prm.dv_real - c * 32);
                    if (grow < N && nc > 0) store_o_row(prm.o, prm.o_fp32, row_elem, vals, c * 32, nc);
                }
            } else {  // the only item of the CTA, or ONE: O released after the stores
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t raw[32];
                    load_o(c, raw);
                    float vals[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) vals[x] = __uint_as_float(raw[x]) * inv_l;
                    const int nc = min(32, prm.dv_real - c * 32);
                    if (grow < N && nc > 0) store_o_row(prm.o, prm.o_fp32, row_elem, vals, c * 32, nc);
                }
                if (PERSIST) release_o();
            }
            if (prm.lse && grow < N) prm.lse[(size_t)wi.bh * N + grow] = (m + log2f(l)) * 0.69314718055994530942f;
        }
    }

    // ---- teardown
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

// A [B, H, n, w] bf16 tensor with element strides st = (batch, head, row)
// and contiguous w, as a 4-D tensor map: w innermost, then the three outer
// dimensions in increasing stride; box = 64 columns (128 bytes, the swizzle
// width) x 128 rows x 1 x 1.  *perm records which of (row, head, batch) each
// outer map dimension holds.  Rows past n read as zeros.
bool make_map(CUtensorMap *map, const void *ptr, int64_t w, int64_t n, int64_t H, int64_t B, const int64_t st[3],
              int *perm)
{
    auto fn = encode_fn();
    if (!fn) return false;
    struct Dim {
        int64_t size, stride;
        int which;
        uint32_t box;
    } dd[3] = {{n, st[2], 0, 128}, {H, st[1], 1, 1}, {B, st[0], 2, 1}};
    for (int i = 1; i < 3; ++i)  // insertion sort by stride, stable
        for (int j = i; j > 0 && dd[j].stride < dd[j - 1].stride; --j) {
            Dim t = dd[j];
            dd[j] = dd[j - 1];
            dd[j - 1] = t;
        }
    cuuint64_t dims[4] = {(cuuint64_t)w, (cuuint64_t)dd[0].size, (cuuint64_t)dd[1].size, (cuuint64_t)dd[2].size};
    cuuint64_t strides[3] = {(cuuint64_t)dd[0].stride * 2, (cuuint64_t)dd[1].stride * 2, (cuuint64_t)dd[2].stride * 2};
    cuuint32_t box[4] = {64, dd[0].box, dd[1].box, dd[2].box};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    *perm = dd[0].which | (dd[1].which << 2) | (dd[2].which << 4);
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count(cudaError_t *e)
{
    int dev = 0, sms = 0;
    if ((*e = cudaGetDevice(&dev)) != cudaSuccess) return 0;
    if ((*e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return 0;
    return std::max(sms, 1);
}

// Workspace layout of a key-range split: o_part [n_split][BH N][DV] fp32, then
// m, l and dq [n_split][BH N] fp32 each (256-byte aligned pieces).
struct SplitLayout {
    size_t o, m, l, d, total;
};
SplitLayout split_layout(const Problem &p, int n_split)
{
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t rows = (size_t)(p.B * p.H * p.N) * (size_t)n_split;
    SplitLayout L;
    L.o = 0;
    L.m = al(rows * (size_t)dv_of(p) * 4);
    L.l = L.m + al(rows * 4);
    L.d = L.l + al(rows * 4);
    L.total = L.d + al(rows * 4);
    return L;
}

// Items of one query tile (ONE): unmasked problems of at most 128 query rows
// per head, and unmasked problems whose two-tile items would fill at most half
// of the SMs.  There twice as many CTAs, each with half the rows and its two
// softmax warpgroups sharing the key tiles, halve the chain of every CTA.  With
// the SMs full, two-tile items win: each K/V tile read from L2 serves 256 rows.
bool one_tile_items(const Problem &p, int sms)
{
    if (p.causal) return false;
    if (p.item_rows) return p.item_rows == BM;
    if (p.N <= BM) return true;
    const int64_t items2 = (p.N + 2 * BM - 1) / (2 * BM) * p.B * p.H;
    return 2 * items2 <= sms;
}

template <int DK, int DV, bool CAUSAL>
cudaError_t launch_typed(const Problem &p, cudaStream_t stream, uint32_t flags, const char **detail,
                         const TcSplit *split = nullptr, void *workspace = nullptr)
{
    CUtensorMap mq, mk, mv;
    const int64_t BH = p.B * p.H, Nk = keys_of(p);
    int64_t sq[3], sk[3], sv[3], so[3];
    strides_of(p, 0, sq);
    strides_of(p, 1, sk);
    strides_of(p, 2, sv);
    strides_of(p, 3, so);
    Params prm;
    // maps of the real widths: the columns a padded head lacks read as zeros,
    // which add nothing to S and leave O's padding columns (never stored) at zero
    if (!make_map(&mq, p.q, p.d, p.N, p.H, p.B, sq, &prm.qperm) || !make_map(&mk, p.k, p.d, Nk, p.H, p.B, sk, &prm.kperm) ||
        !make_map(&mv, p.v, dv_of(p), Nk, p.H, p.B, sv, &prm.vperm)) {
        *detail = "cuTensorMapEncodeTiled failed or is unavailable";
        return cudaErrorInvalidValue;
    }
    prm.N = (int)p.N;
    prm.Nk = (int)Nk;
    prm.H = (int)p.H;
    prm.BH = (int)BH;
    cudaError_t e = cudaSuccess;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    const bool one = one_tile_items(p, sms);
    const int item_rows = one ? BM : 2 * BM;
    prm.n_qblocks = (int)((p.N + item_rows - 1) / item_rows);
    prm.n_items = (int)(prm.n_qblocks * BH);
    {   // causal item order: as many heads per group as keep their K and V within
        // half of L2 (a head's K/V stays there while its query blocks run)
        int dev = 0, l2 = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            l2 = 0;
        const int64_t kv_head = Nk * (int64_t)(DK + DV) * 2;
        const int64_t g = l2 > 0 ? (int64_t)l2 / 2 / std::max<int64_t>(kv_head, 1) : BH;
        prm.hgroup = (int)std::max<int64_t>(1, std::min<int64_t>(g, BH));
    }
    prm.n_kv = (int)((Nk + BN - 1) / BN);
    prm.scale_log2 = p.scale * 1.4426950408889634f;
    prm.causal = CAUSAL;
    const bool inject = (flags & FA_FLAG_TEST_SKIP_KV_LOAD) != 0;
    prm.skip_load = inject ? 1 : -1;
    // 2 s is far above any legitimate wait; the fault-injection test uses 20 ms
    prm.wait_limit_ns = inject ? 20000000ull : 2000000000ull;
    prm.o = p.o;
    prm.os_b = so[0];
    prm.os_h = so[1];
    prm.os_n = so[2];
    prm.lse = p.lse;
    prm.o_fp32 = p.o_dtype == 1;
    prm.dv_real = (int)dv_of(p);
    prm.n_split = 1;
    prm.kv_per = prm.n_kv;
    prm.o_part = prm.m_part = prm.l_part = prm.d_part = nullptr;
    if (split && split->n_split > 1) {
        const SplitLayout L = split_layout(p, split->n_split);
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        prm.n_split = split->n_split;
        prm.kv_per = split->kv_per;
        prm.o_part = reinterpret_cast<float *>(ws + L.o);
        prm.m_part = reinterpret_cast<float *>(ws + L.m);
        prm.l_part = reinterpret_cast<float *>(ws + L.l);
        prm.d_part = reinterpret_cast<float *>(ws + L.d);
        prm.n_items *= prm.n_split;
    }
    // Short unmasked items (64 key tiles or fewer): one persistent CTA per SM
    // loops over them, so an item's prologue (query loads, first S MMA) and
    // epilogue overlap its neighbours' work (multi-head workload +2.5 %).  Long
    // items gain nothing from that, and long items of unequal cost (causal)
    // balance best one per CTA, handed out by the hardware as SMs free up
    // (measured: persistence with alternating-direction rounds gave the causal
    // workload -1 %, the peaked one -2 %).  Short causal items, when there are
    // more of them than SMs, gain more from the overlap than they lose in
    // balance: at most 2048 key-tile columns (16 key tiles at d = 128, 32 at
    // d = 64) measured +4 to +31 % on 512-4096-key problems.
    const bool persist = prm.n_split == 1 && (CAUSAL ? prm.n_items > sms && prm.n_kv * std::max(DK, DV) <= 2048
                                                     : prm.n_kv <= 64);
    auto kern = prm.n_split > 1 ? (one ? fa_tc_kernel<DK, DV, CAUSAL, false, !CAUSAL, !CAUSAL>
                                       : fa_tc_kernel<DK, DV, CAUSAL, false, !CAUSAL, false>)
                : persist       ? (one ? fa_tc_kernel<DK, DV, CAUSAL, true, false, !CAUSAL>
                                       : fa_tc_kernel<DK, DV, CAUSAL, true, false, false>)
                                : (one ? fa_tc_kernel<DK, DV, CAUSAL, false, false, !CAUSAL>
                                       : fa_tc_kernel<DK, DV, CAUSAL, false, false, false>);
    const uint32_t smem_bytes = one ? Cfg<DK, DV, true>::SMEM_BYTES : Cfg<DK, DV>::SMEM_BYTES;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    int grid = prm.n_items;
    if (persist) grid = std::min(prm.n_items, sms);
    kern<<<(unsigned)grid, NUM_THREADS, smem_bytes, stream>>>(mq, mk, mv, prm);
    if ((e = cudaGetLastError()) != cudaSuccess || prm.n_split == 1) return e;
    return launch_combine(prm.o_part, prm.m_part, prm.l_part, prm.d_part, p.o, p.o_dtype == 1, p.lse, BH, p.N, DV,
                          prm.n_split, stream);
}

template <int DK, int DV>
cudaError_t launch_dims(const Problem &p, cudaStream_t stream, uint32_t flags, const char **detail,
                        const TcSplit *split = nullptr, void *workspace = nullptr)
{
    return p.causal ? launch_typed<DK, DV, true>(p, stream, flags, detail)
                    : launch_typed<DK, DV, false>(p, stream, flags, detail, split, workspace);
}

}  // namespace

// Head widths the kernel covers: 64 and 128, and any narrower multiple of 8
// (16-byte rows for TMA), padded up to 64 or 128 with zero columns.
inline bool tc_width(int64_t w) { return w >= 8 && w <= 128 && w % 8 == 0; }
inline int tc_padded(int64_t w) { return w <= 64 ? 64 : 128; }

bool tc_supported(const Problem &p)
{
    const int64_t dv = dv_of(p);
    if (p.in_dtype != 0 || !tc_width(p.d) || !tc_width(dv) || !(p.scale > 0.f)) return false;
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    if (!(al16(p.q) && al16(p.k) && al16(p.v) && al16(p.o))) return false;
    // TMA: every stride a non-zero multiple of 16 bytes; O rows start 16-byte aligned
    const int64_t o_elt = p.o_dtype == 1 ? 4 : 2;
    for (int t = 0; t < 4; ++t) {
        int64_t st[3];
        strides_of(p, t, st);
        const int64_t elt = t == 3 ? o_elt : 2;
        for (int i = 0; i < 3; ++i)
            if (st[i] <= 0 || (st[i] * elt) % 16 != 0) return false;
    }
    return true;
}

cudaError_t launch_tc(const Problem &p, cudaStream_t stream, uint32_t flags, const char **detail)
{
    const int dk = tc_padded(p.d), dv = tc_padded(dv_of(p));
    if (dk == 128) return dv == 128 ? launch_dims<128, 128>(p, stream, flags, detail)
                                    : launch_dims<128, 64>(p, stream, flags, detail);
    return dv == 128 ? launch_dims<64, 128>(p, stream, flags, detail) : launch_dims<64, 64>(p, stream, flags, detail);
}

// Flash-decoding style split for problems with few work items: unmasked, O
// contiguous, at most one wave of (item, split) CTAs, two key tiles or more
// per split, 16 splits at most (the combine kernel's limit).
int tc_item_rows(const Problem &p)
{
    cudaError_t e = cudaSuccess;
    const int sms = sm_count(&e);
    return one_tile_items(p, e == cudaSuccess ? sms : 0) ? BM : 2 * BM;
}

TcSplit tc_split_plan(const Problem &p)
{
    TcSplit sp{1, 0, 0};
    if (p.causal || !tc_supported(p)) return sp;
    const int64_t dv = dv_of(p);
    if (tc_padded(p.d) != p.d || tc_padded(dv) != dv) return sp;  // the merge writes whole 64/128-column rows
    int64_t os[3];
    strides_of(p, 3, os);
    if (os[2] != dv || os[1] != p.N * dv || os[0] != p.H * p.N * dv) return sp;  // combine writes contiguous O
    cudaError_t e = cudaSuccess;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return sp;
    const int64_t item_rows = one_tile_items(p, sms) ? BM : 2 * BM;
    const int64_t items = (p.N + item_rows - 1) / item_rows * p.B * p.H;
    const int64_t n_kv = (keys_of(p) + BN - 1) / BN;
    if (2 * items > sms || n_kv < 4) return sp;
    int64_t n = std::min<int64_t>({16, sms / items, n_kv / 2});
    if (n < 2) return sp;
    const int64_t per = (n_kv + n - 1) / n;
    n = (n_kv + per - 1) / per;
    if (n < 2) return sp;
    sp.n_split = (int)n;
    sp.kv_per = (int)per;
    sp.workspace_bytes = split_layout(p, sp.n_split).total;
    return sp;
}

cudaError_t launch_tc_split(const Problem &p, const TcSplit &sp, void *workspace, cudaStream_t stream, const char **detail)
{
    const int64_t dv = dv_of(p);  // not padded: tc_split_plan splits only 64 and 128
    if (p.d == 128) return dv == 128 ? launch_dims<128, 128>(p, stream, 0, detail, &sp, workspace)
                                     : launch_dims<128, 64>(p, stream, 0, detail, &sp, workspace);
    return dv == 128 ? launch_dims<64, 128>(p, stream, 0, detail, &sp, workspace)
                     : launch_dims<64, 64>(p, stream, 0, detail, &sp, workspace);
}

cudaError_t tc_error_word_ptr(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_tc_error_word);
}

}  // namespace fa
