// Flash-attention backward on the sm_103a tensor cores (bf16 in, fp32 accumulate).
//
// Method: "xtrain docs/13-flash-attention.md", section "什么是 flash-attention"
// (recompute s_ij = scale Q_i.K_j and p_ij = exp(s_ij - L_i), dp_ij = dO_i.V_j,
// ds_ij = p_ij (dp_ij - D_i) scale, then dQ_i += ds_ij K_j, dK_j += ds_ij Q_i,
// dV_j += p_ij dO_i) with D_i = dO_i.O_i from the pre-pass (design decision ③).
//
// GB300 design: the key-block-owned backward that the page names as its
// follow-up, on tcgen05:
//   * persistent CTAs, one per SM; a work item is 128 keys of one head (claimed from a
//     per-launch counter); K_j and V_j are loaded once per item by TMA and dK_j, dV_j
//     accumulate in TMEM (128 lanes = keys, hd fp32 columns each) over every 64-row
//     query tile at or below the diagonal, then go straight to global memory;
//   * warp 8 streams Q_i, dO_i (TMA, 128-byte swizzle) with -L_i*log2(e) and
//     D_i (bulk copies) through a ring;
//   * warp 9 (one thread) issues, per query tile:
//       S^T  = K_j Q_i^T            (M=128 keys, N=64 rows, K=hd; A = K_j kept in TMEM)
//       dP^T = V_j dO_i^T           (M=128, N=64, K=hd)            -> TMEM
//       dV  += P^T dO_i             (A = P^T bf16 in TMEM, B = dO_i MN-major)
//       dK  += dS^T Q_i             (A = dS^T bf16 in TMEM, B = Q_i MN-major)
//       dQ^T = K_j^T dS^T           (M=hd, N=64, K=128 keys; B = dS^T in smem) -> TMEM
//     Operands kept in TMEM spare shared-memory bandwidth, which bounds this kernel;
//   * warps 0-3 (thread = key) turn S^T, dP^T into P^T (bf16, back into the
//     S^T columns) and dS^T (bf16, swizzled smem);
//   * warps 4-7 (thread = hd index) read dQ^T from TMEM, stage it as a
//     row-major fp32 [64][hd] tile in shared memory (one contiguous block of
//     the [S][hd] accumulator) and add it into global memory with a single
//     TMA bulk reduce-add; a conversion kernel writes dQ afterwards.
// TMEM map (512 columns): dK [0,hd) dV [hd,2hd) S^T [2hd,2hd+64) dP^T [2hd+64,2hd+128)
//                         dQ^T [2hd+128,2hd+192) K_j [2hd+192,2hd+192+hd/2).
// For hd = 64 the dQ^T MMA still runs with M = 128; lanes 64-127 hold
// products of V and are never read.
// Without the fused dQ (the deterministic variant) the dQ^T columns hold a second
// S^T buffer, and at hd = 64 the columns past K_j do: tiles alternate between the
// two, and S^T of the next tile is issued before this tile's dV, so the key warps
// do not wait for it.  At hd = 64 with the fused dQ a second dP^T buffer follows
// (columns [416, 480)), so the next tile's dP^T is issued before this tile's dK.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <atomic>

#include "dropout.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace xfa {
namespace {

constexpr int BN = 128;       // keys per CTA (MMA M)
constexpr int BM = 64;        // query rows per tile (MMA N of S^T / dP^T)
// query-tile (Q, dO, L, D) ring stages; with dropout at hd = 128 two, to make room for the keep bits
template <int HD, bool DROP>
constexpr int ring_depth() { return HD == 128 ? (DROP ? 2 : 3) : 4; }
constexpr int kThreads = 320;
constexpr int kWarpTma = 8, kWarpMma = 9;
// With dropout: 20 warps.  Warps 12-19 (two warpgroups, two warps per SM sub-partition: the draw
// is bound by the integer multiplier, which one warp per sub-partition does not keep busy) draw
// the keep bits of every (key, query row) of the coming query tiles into shared memory (MSB
// stages), so the key-row warps only read them; warps 10-11 are idle.  A 640-thread launch gets 96
// registers a thread: the key-row warpgroup grows to 184 and the readout warpgroup to 128, the
// TMA/MMA/idle warpgroup and the mask warpgroups shrink to 56 (184 + 128 + 56 + 2 x 56 = 480 per
// lane of a warpgroup, 96 x 5).
constexpr int kMaskWarps = 8;
constexpr int kWarpMask0 = 12;
constexpr int kThreadsDrop = (kWarpMask0 + kMaskWarps) * 32;
constexpr int MSB = 4;   // keep-bit stages (query tiles)

struct MaskBars {
    uint64_t full[MSB];    // keep bits of a query tile written (one arrival per mask warp)
    uint64_t empty[MSB];   // read by the key-row warps (one arrival per warp)
};
constexpr int kHeadBundle = 4;   // heads scheduled together at long S (L2 reuse of inputs and dQ accumulator)

template <int HD, bool DROP = false>
struct Cfg {
    static constexpr int NSQ = ring_depth<HD, DROP>();
    static constexpr int SUB = HD / 64;
    static constexpr int KV_SUB = BN * 128;             // 128 rows x 128 B
    static constexpr int Q_SUB = BM * 128;              // 64 rows x 128 B
    static constexpr int KV_BYTES = BN * HD * 2;
    static constexpr int Q_BYTES = BM * HD * 2;
    static constexpr int DS_BYTES = BN * BM * 2;        // dS^T: 128 keys x 64 rows bf16 = 128 B rows
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KV_BYTES;
    static constexpr int OFF_Q = 2 * KV_BYTES;
    static constexpr int OFF_DO = OFF_Q + NSQ * Q_BYTES;
    static constexpr int OFF_DS = OFF_DO + NSQ * Q_BYTES;
    static constexpr int OFF_DQ = OFF_DS + 2 * DS_BYTES;  // fp32 dQ tile [64 rows][hd] staged for the bulk reduce
    static constexpr int OFF_LD = OFF_DQ + BM * HD * 4;   // per stage: Lg[64], D[64]
    // dropout: keep bits [stage][key] x 64 query rows, then their barriers
    static constexpr int OFF_MASK = OFF_LD + NSQ * 2 * BM * 4;
    static constexpr int OFF_MBAR = OFF_MASK + (DROP ? MSB * BN * 8 : 0);
    static constexpr int OFF_BAR = OFF_MBAR + (DROP ? 128 : 0);
    static constexpr int SMEM = OFF_BAR + 256 + 1024;   // barriers + alignment slack
    // TMEM columns: dK, dV accumulators; S^T (P^T bf16 written back into its first 32 columns);
    // dP^T (dS^T bf16 written back into its first 32 columns); dQ^T; K_j as a bf16 A operand.
    static constexpr uint32_t COL_DK = 0, COL_DV = HD, COL_S = 2 * HD, COL_DP = 2 * HD + 64,
                              COL_DQ = 2 * HD + 128, COL_KT = 2 * HD + 192, COL_S2 = COL_KT + HD / 2;
    static constexpr uint32_t TMEM_COLS = 512;
    // S^T buffers: query tiles alternate between two when there is room -- without the fused dQ
    // (the dQ^T columns are free) or at hd = 64 (columns past K_j) -- else they share one.
    template <bool FUSED_DQ>
    static __host__ __device__ constexpr bool two_s() { return !FUSED_DQ || COL_S2 + 64 <= TMEM_COLS; }
    template <bool FUSED_DQ>
    static __device__ __forceinline__ uint32_t col_s(uint32_t i)
    {
        return two_s<FUSED_DQ>() && (i & 1) ? (FUSED_DQ ? COL_S2 : COL_DQ) : COL_S;
    }
    // dP^T buffers: with the fused dQ at hd = 64 there is room for a second one past the second
    // S^T, and tiles alternate between the two, so the next tile's dP^T is issued before this
    // tile's dK (which reads dS^T out of this tile's dP^T columns).
    static constexpr uint32_t COL_DP2 = COL_S2 + 64;
    template <bool FUSED_DQ>
    static __host__ __device__ constexpr bool two_dp() { return FUSED_DQ && HD == 64 && COL_DP2 + 64 <= TMEM_COLS; }
    template <bool FUSED_DQ>
    static __device__ __forceinline__ uint32_t col_dp(uint32_t i)
    {
        return two_dp<FUSED_DQ>() && (i & 1) ? COL_DP2 : COL_DP;
    }
};

constexpr int kMaxRing = 4;

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[kMaxRing], q_empty[kMaxRing];
    // ds_full[b]: dS of a tile written (key warps) and, with the fused dQ at hd = 64, the previous
    // tile's dQ^T read out of TMEM (readout warps) -- one barrier for the MMA warp to wait on before
    // the tile's dK, next dP^T and dQ^T.  At hd = 128 the readout signals dq_empty instead: there
    // its staging is long enough that tying dK to it would hold up the whole chain.
    uint64_t s_full[2], p_full, ds_full[2], ds_empty[2];
    uint64_t kt_full, dp_full[2], dq_full, dq_empty, done, drain;
    uint64_t dk_read;                      // the readout warps have read the item's dK out of TMEM
    uint64_t item_full[2], item_empty[2];  // work-item ids posted by the TMA warp, read by the others
    int item_id[2];                        // the posted ids (-1: no more work)
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void fail(Bars *b, int *status)
{
    b->abort = 1;
    record_status(status, XFA_ERR_TIMEOUT);
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, Bars *b, int *status)
{
    bool ok = mbar_wait(bar, parity, &b->abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) fail(b, status);
    return ok;
}

// Epilogue of one 128-row accumulator (dK or dV) straight to global memory: thread = row of the
// key tile (TMEM lane), its hd fp32 columns converted to bf16 and written as 16-byte stores; rows
// past S are not written.
template <int HD>
__device__ __forceinline__ void store_rows_global(uint32_t t_row, __nv_bfloat16 *dst, bool valid)
{
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
        uint32_t o[32];
        tmem_ld32(t_row + c, o);
        tmem_wait_ld();
        reg_fence32(o);
        if (valid) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]), __uint_as_float(o[8 * v + 1]));
                w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3]));
                w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5]));
                w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7]));
                d4[v] = w;
            }
        }
    }
}

// The next work item for a consumer warp: waits until the TMA warp has posted it in ring entry
// k & 1, reads it and releases the entry (one arrival per warp).  -1: no more work, or the
// wait gave up (then ok is false).
__device__ __forceinline__ int take_item(Bars *b, int k, int *status, bool &ok)
{
    const int e = k & 1;
    if (!(ok = warp_wait(&b->item_full[e], (k >> 1) & 1, b, status))) return -1;
    const int item = *reinterpret_cast<volatile int *>(&b->item_id[e]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&b->item_empty[e]);
    return item;
}

// C[M=128, N=64] = A[128 rows x hd] * B[64 rows x hd]^T, both K-major (hd contiguous);
// descriptors of the tile bases, advanced per 16-wide K step.
template <int HD>
__device__ __forceinline__ void issue_rows_dot(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc)
{
    constexpr uint32_t idesc = idesc_bf16(BN, BM, false, false);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
        const uint32_t k_off = (ks % 4) * 32;
        mma_ss(d_tmem, sdesc_advance(a_desc, (ks / 4) * Cfg<HD>::KV_SUB + k_off),
               sdesc_advance(b_desc, (ks / 4) * Cfg<HD>::Q_SUB + k_off), idesc, ks > 0);
    }
}

// S^T[M=128 keys, N=64 rows] = K_j (A: bf16 pairs in TMEM, hd along the columns) * Q_i^T (B: K-major smem).
template <int HD>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t k_tmem, uint64_t q_desc, uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks)
        mma_ts(d_tmem, k_tmem + ks * 8, sdesc_advance(q_desc, (ks / 4) * Cfg<HD>::Q_SUB + (ks % 4) * 32), idesc,
               ks > 0 ? 1u : 0u);
}

// FUSED_DQ: dQ^T is formed here and summed into the fp32 accumulator (bulk reduce-add);
// otherwise dQ is left to the query-tile pass (tc_dq.cu) and this kernel does dK, dV only.
// DROP: dropout on the attention probabilities (fused only): dV takes P o C and dS is
// formed from C o dP, with C re-drawn from (seed, flat index).
template <int HD, bool FUSED_DQ, bool DROP>
__global__ void __launch_bounds__(DROP ? kThreadsDrop : kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const float *__restrict__ Lg, const float *__restrict__ Dg, float *__restrict__ dq_acc,
                  __nv_bfloat16 *__restrict__ dK, __nv_bfloat16 *__restrict__ dV, int bh, int S, int S_pad,
                  float scale, float scale_log2, int *status, const DropParams drop, int bundle_heads,
                  unsigned *__restrict__ next_item)
{
    using C = Cfg<HD, DROP>;
    constexpr int NSQ = C::NSQ;
    constexpr bool TWO_S = C::template two_s<FUSED_DQ>();
    constexpr bool TWO_DP = C::template two_dp<FUSED_DQ>();
    static_assert(!TWO_DP || TWO_S, "the early dP^T relies on the early S^T's wait for the query stage");
    static_assert(NSQ <= kMaxRing && sizeof(Bars) <= 256, "barrier block");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    float *ld_s = reinterpret_cast<float *>(smem + C::OFF_LD);
    float *dq_stage = reinterpret_cast<float *>(smem + C::OFF_DQ);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Persistent CTAs: at most one per SM, each taking work items -- the 128 keys of one key tile
    // of one head -- from a shared counter (next_item, zeroed before the launch) until the list
    // is exhausted: greedy scheduling without a CTA teardown and launch between items.  The list
    // runs heads in bundles of bundle_heads (see head_bundle: at long S the inputs and the dQ
    // accumulator of the heads in flight stay in L2) and, within a bundle, the key tiles with the
    // most query tiles first.  The TMA warp claims an item and posts its id to the other warps
    // through a two-entry ring.  Every per-tile barrier phase, ring stage and dS buffer follows
    // the CTA's running count of query tiles (gi), so the query ring streams on from one item into
    // the next; K and V of the next item load once the current item's MMAs are done with them.
    const int nkt = (S + BN - 1) / BN;
    const int n_items = nkt * bh;
    const int nq_total = (S + BM - 1) / BM;
    struct Item {
        int head, j0, it0, n;   // head, first key, first query tile at or below the diagonal, tiles
    };
    auto item_of = [&](int item) {
        const int bundle = item / (nkt * bundle_heads);
        const int g = min(bundle_heads, bh - bundle * bundle_heads);
        const int idx = item - bundle * nkt * bundle_heads;
        Item w;
        w.head = bundle * bundle_heads + idx % g;
        w.j0 = (idx / g) * BN;
        w.it0 = w.j0 / BM;
        w.n = nq_total - w.it0;   // >= 1
        return w;
    };

    if (threadIdx.x == 0) {
        mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < NSQ; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            // one arrival per key warp (+ one per dQ readout warp at hd = 64)
            mbar_init(&bars->ds_full[b], 4 + (FUSED_DQ && HD == 64 ? HD / 32 : 0));
            mbar_init(&bars->ds_empty[b], 1);
            mbar_init(&bars->item_full[b], 1);
            // MMA warp, four key warps, four readout warps (+ the keep-bit warps)
            mbar_init(&bars->item_empty[b], 9 + (DROP ? kMaskWarps : 0));
        }
        mbar_init(&bars->s_full[0], 1);
        mbar_init(&bars->s_full[1], 1);
        mbar_init(&bars->p_full, 4);
        mbar_init(&bars->kt_full, 4);
        mbar_init(&bars->dp_full[0], 1);
        mbar_init(&bars->dp_full[1], 1);
        mbar_init(&bars->dq_full, 1);
        mbar_init(&bars->dq_empty, HD / 32);   // one arrival per readout warp (hd = 128)
        mbar_init(&bars->done, 1);
        mbar_init(&bars->dk_read, 4);         // one arrival per readout warp
        mbar_init(&bars->drain, 1);
        if (DROP) {
            MaskBars *mb = reinterpret_cast<MaskBars *>(smem + C::OFF_MBAR);
            for (int s = 0; s < MSB; ++s) {
                // drawn: one arrival per keep-bit warp; cached: one bulk copy (arrival + bytes)
                mbar_init(&mb->full[s], drop.keep_in ? 1 : kMaskWarps);
                mbar_init(&mb->empty[s], 4);
            }
        }
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    MaskBars *mbars = reinterpret_cast<MaskBars *>(smem + C::OFF_MBAR);
    const uint32_t *mask_s = reinterpret_cast<const uint32_t *>(smem + C::OFF_MASK);

    // Roles by warpgroup (with dropout every warpgroup first resizes its registers, all four warps
    // together): warps 8-11 the TMA and MMA warps (and two idle ones), 12-19 the keep-bit warps,
    // 0-3 the key-row warps, 4-7 the dQ readout warps.
    if (warp >= 8 && warp < 12) {
        if (DROP) regs_decrease<56>();
        if (warp == kWarpTma) {
            if (lane == 0) {
                prefetch_tensormap(&tm_k);
                prefetch_tensormap(&tm_v);
                prefetch_tensormap(&tm_q);
                prefetch_tensormap(&tm_do);
                uint32_t gt = 0;                      // query tiles issued
                uint32_t last[kMaxRing] = {};         // 1 + last tile issued per stage
                int kv_loads = 0;
                bool ok = true;
                for (int kc = 0; ok; ++kc) {          // kc: items claimed, posted in ring entry kc & 1
                    const int e = kc & 1;
                    if (kc >= 2 && !(ok = mbar_wait(&bars->item_empty[e], ((kc >> 1) + 1) & 1, &bars->abort))) break;
                    int item = (int)atomicAdd(next_item, 1u);
                    if (item >= n_items) item = -1;
                    *reinterpret_cast<volatile int *>(&bars->item_id[e]) = item;
                    mbar_arrive(&bars->item_full[e]);
                    if (item < 0) break;
                    const Item w = item_of(item);
                    // K, V of this item: their buffers are free once the previous item's MMAs are done
                    if (kc > 0 && !(ok = mbar_wait(&bars->done, (kc - 1) & 1, &bars->abort))) break;
                    mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KV_BYTES);
                    for (int s = 0; s < C::SUB; ++s) {
                        tma_load_3d(smem + C::OFF_K + s * C::KV_SUB, &tm_k, &bars->kv_full, s * 64, w.j0, w.head);
                        tma_load_3d(smem + C::OFF_V + s * C::KV_SUB, &tm_v, &bars->kv_full, s * 64, w.j0, w.head);
                    }
                    ++kv_loads;
                    for (int it = 0; it < w.n; ++it) {
                        const uint32_t gi = gt + it;
                        const int st = gi % NSQ;
                        if (gi >= NSQ && !(ok = mbar_wait(&bars->q_empty[st], ((gi / NSQ) + 1) & 1, &bars->abort))) break;
                        const int i0 = (w.it0 + it) * BM;
                        mbar_arrive_expect_tx(&bars->q_full[st], 2 * C::Q_BYTES + 2 * BM * 4);
                        for (int s = 0; s < C::SUB; ++s) {
                            tma_load_3d(smem + C::OFF_Q + st * C::Q_BYTES + s * C::Q_SUB, &tm_q, &bars->q_full[st],
                                        s * 64, i0, w.head);
                            tma_load_3d(smem + C::OFF_DO + st * C::Q_BYTES + s * C::Q_SUB, &tm_do, &bars->q_full[st],
                                        s * 64, i0, w.head);
                        }
                        float *ld = ld_s + st * 2 * BM;
                        bulk_load(ld, Lg + (size_t)w.head * S_pad + i0, BM * 4, &bars->q_full[st]);
                        bulk_load(ld + BM, Dg + (size_t)w.head * S_pad + i0, BM * 4, &bars->q_full[st]);
                        last[st] = gi + 1;
                    }
                    gt += w.n;
                }
                if (!ok) fail(bars, status);
                // Never leave the CTA with copies in flight: wait for the last load of K/V and of each stage.
                if (kv_loads > 0) mbar_wait(&bars->kv_full, (kv_loads - 1) & 1, nullptr);
                for (int st = 0; st < NSQ; ++st)
                    if (last[st]) mbar_wait(&bars->q_full[st], ((last[st] - 1) / NSQ) & 1, nullptr);
            }
        } else if (warp == kWarpMma) {
            // The whole warp runs the issue loop (converged, descriptors warp-uniform);
            // one elected lane issues the tcgen05 instructions.
            const bool leader = elect_one();
            const uint32_t k_s = smem_u32(smem + C::OFF_K), v_s = smem_u32(smem + C::OFF_V);
            const uint32_t q_s = smem_u32(smem + C::OFF_Q), do_s = smem_u32(smem + C::OFF_DO);
            const uint32_t ds_s = smem_u32(smem + C::OFF_DS);
            // K-major views (hd contiguous) for dP^T = V dO^T and the B operand Q_i of S^T
            const uint64_t v_km = sdesc_sw128(v_s, 16, 1024);
            const uint64_t q_km = sdesc_sw128(q_s, 16, 1024), do_km = sdesc_sw128(do_s, 16, 1024);
            // MN-major views: B = dO_i / Q_i for dV / dK, A = K_j^T for dQ^T; dS^T as K-major A / MN-major B
            const uint64_t do_mn = sdesc_sw128(do_s, C::Q_SUB, 1024), q_mn = sdesc_sw128(q_s, C::Q_SUB, 1024);
            const uint64_t k_mn = sdesc_sw128(k_s, C::KV_SUB, 1024);
            const uint64_t ds_mn = sdesc_sw128(ds_s, C::DS_BYTES, 1024);
            constexpr uint32_t idesc_acc = idesc_bf16(BN, HD, false, true);    // dV, dK: B MN-major
            constexpr uint32_t idesc_dq = idesc_bf16(128, BM, true, true);     // dQ^T: A, B MN-major
            constexpr uint32_t idesc_s = idesc_bf16(BN, BM, false, false);     // S^T: A = K_j from TMEM
            uint32_t gt = 0;   // query tiles of earlier items
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = take_item(bars, k, status, ok);
                if (item < 0) break;
                const int n = item_of(item).n;
                const int st0 = gt % NSQ;
                ok = warp_wait(&bars->kv_full, k & 1, bars, status) && warp_wait(&bars->kt_full, k & 1, bars, status) &&
                     warp_wait(&bars->q_full[st0], (gt / NSQ) & 1, bars, status);
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
                    // the S^T / dP^T columns last held the previous item's final P^T / dS^T, read by
                    // its dV / dK MMAs issued before (in order)
                    issue_s<HD>(tmem + C::template col_s<FUSED_DQ>(gt), tmem + C::COL_KT,
                                sdesc_advance(q_km, st0 * C::Q_BYTES), idesc_s);
                    tc_commit(&bars->s_full[TWO_S ? (gt & 1) : 0]);
                    issue_rows_dot<HD>(tmem + C::template col_dp<FUSED_DQ>(gt), v_km, sdesc_advance(do_km, st0 * C::Q_BYTES));
                    tc_commit(&bars->dp_full[TWO_DP ? (gt & 1) : 0]);
                }
                __syncwarp();
                for (int it = 0; ok && it < n; ++it) {
                    const uint32_t gi = gt + it;
                    const int b = gi & 1, st = gi % NSQ;
                    const uint32_t ph2 = (gi >> 1) & 1;
                    const uint32_t qoff = st * C::Q_BYTES, dsoff = b * C::DS_BYTES;
                    const int nx = it + 1;
                    const uint32_t gn = gi + 1;
                    const int stn = gn % NSQ;
                    // Next S^T.  With two S^T buffers it goes first, into the other one, so that it
                    // does not queue behind this tile's work (that buffer's P^T, tile gi - 1, was read by
                    // the dV MMA issued one iteration ago, and the in-order pipe runs that MMA first).
                    // With one buffer it follows this tile's dV, which reads P^T from the same columns.
                    const bool s_first = TWO_S && nx < n;
                    if (s_first) {
                        if (!(ok = warp_wait(&bars->q_full[stn], (gn / NSQ) & 1, bars, status))) break;
                        tc_fence_after_sync();
                        if (leader) {
                            issue_s<HD>(tmem + C::template col_s<FUSED_DQ>(gn), tmem + C::COL_KT, sdesc_advance(q_km, stn * C::Q_BYTES),
                                        idesc_s);
                            tc_commit(&bars->s_full[gn & 1]);
                        }
                        __syncwarp();
                    }
                    // dV += P^T dO_i  (P^T: bf16 in the first columns of this tile's S^T).  The item's
                    // first dV overwrites the accumulator, which the key warps have read out before
                    // they wrote this P^T.
                    if (!(ok = warp_wait(&bars->p_full, gi & 1, bars, status))) break;
                    tc_fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < BM / 16; ++ks)
                            mma_ts(tmem + C::COL_DV, tmem + C::template col_s<FUSED_DQ>(gi) + ks * 8,
                                   sdesc_advance(do_mn, qoff + ks * 2048), idesc_acc, (it > 0 || ks > 0) ? 1u : 0u);
                    }
                    __syncwarp();
                    if (TWO_DP && nx < n) {
                        // next dP^T into the other buffer: its dS^T (tile gi - 1) was read by the dK MMA
                        // issued one iteration ago; its query stage was waited for with the next S^T
                        if (leader) {
                            issue_rows_dot<HD>(tmem + C::template col_dp<FUSED_DQ>(gn), v_km, sdesc_advance(do_km, stn * C::Q_BYTES));
                            tc_commit(&bars->dp_full[gn & 1]);
                        }
                        __syncwarp();
                    }
                    if (!TWO_S && nx < n) {   // next S^T: its columns are free once the dV MMA above has read P^T
                        if (!(ok = warp_wait(&bars->q_full[stn], (gn / NSQ) & 1, bars, status))) break;
                        tc_fence_after_sync();
                        if (leader) {
                            issue_s<HD>(tmem + C::COL_S, tmem + C::COL_KT, sdesc_advance(q_km, stn * C::Q_BYTES), idesc_s);
                            tc_commit(&bars->s_full[0]);
                        }
                        __syncwarp();
                    }
                    // dS^T is in TMEM (first columns of dP^T) and in smem: dK first (reads the TMEM copy),
                    // then the next dP^T may overwrite those columns.  The item's first dK overwrites the
                    // accumulator: the readout warps must have read the previous item's dK out of it.
                    // With the fused dQ at hd = 64 the same barrier also says that the readout warps have
                    // read the previous tile's dQ^T out of TMEM, so this tile's dQ^T may overwrite it.
                    if (!(ok = warp_wait(&bars->ds_full[b], ph2, bars, status))) break;
                    if (it == 0 && k > 0 && !(ok = warp_wait(&bars->dk_read, (k - 1) & 1, bars, status))) break;
                    tc_fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < BM / 16; ++ks)
                            mma_ts(tmem + C::COL_DK, tmem + C::template col_dp<FUSED_DQ>(gi) + ks * 8,
                                   sdesc_advance(q_mn, qoff + ks * 2048), idesc_acc, (it > 0 || ks > 0) ? 1u : 0u);
                        tc_commit(&bars->q_empty[st]);
                        if (!TWO_DP && nx < n) {
                            issue_rows_dot<HD>(tmem + C::COL_DP, v_km, sdesc_advance(do_km, stn * C::Q_BYTES));
                            tc_commit(&bars->dp_full[0]);
                        }
                    }
                    __syncwarp();
                    if (FUSED_DQ) {
                        if (HD == 128 && gi > 0 && !(ok = warp_wait(&bars->dq_empty, (gi - 1) & 1, bars, status)))
                            break;
                        tc_fence_after_sync();
                        if (leader) {
#pragma unroll
                            for (int ks = 0; ks < BN / 16; ++ks)
                                mma_ss(tmem + C::COL_DQ, sdesc_advance(k_mn, ks * 2048),
                                       sdesc_advance(ds_mn, dsoff + ks * 2048), idesc_dq, ks > 0 ? 1u : 0u);
                            tc_commit(&bars->dq_full);
                            if (HD == 128) tc_commit(&bars->ds_empty[b]);
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                if (leader) tc_commit(&bars->done);   // every MMA of this item (K, V, the accumulators)
                __syncwarp();
                gt += n;
            }
            if (leader) {
                tc_commit(&bars->drain);
                mbar_wait(&bars->drain, 0, nullptr);
            }
            __syncwarp();
        }
    } else if (warp >= 12) {
        if (DROP) {
            regs_decrease<56>();
            // keep bits (dropout) of every query tile, in the order the key-row warps consume them, as
            // two 128-word rows per stage (row m: bit c of word r = decision of (row i0 + 32m + c, key r)).
            uint32_t *mask_w = reinterpret_cast<uint32_t *>(smem + C::OFF_MASK);
            const int mw = warp - kWarpMask0;
            uint32_t nm = 0;   // stages filled
            bool ok = true;
            if (drop.keep_in) {
                // cached by the forward in the same order (keep_word): one thread copies each tile's
                // 1 KB with a bulk copy, up to MSB tiles ahead; the other keep-bit warps only take items
                const bool lead = mw == 0;
                const bool issuer = lead && elect_one();
                const int issuer_lane = lead ? __ffs(__ballot_sync(0xffffffffu, issuer)) - 1 : 0;
                uint32_t last[MSB] = {};   // 1 + last tile copied per stage
                for (int k = 0; ok; ++k) {
                    const int item = take_item(bars, k, status, ok);
                    if (item < 0) break;
                    const Item w = item_of(item);
                    if (issuer) {
                        for (int it = 0; it < w.n; ++it, ++nm) {
                            const uint32_t st = nm % MSB;
                            if (nm >= MSB && !(ok = mbar_wait(&mbars->empty[st], ((nm / MSB) + 1) & 1, &bars->abort))) break;
                            mbar_arrive_expect_tx(&mbars->full[st], 2 * BN * 4);
                            bulk_load(mask_w + st * 2 * BN,
                                      drop.keep_in + keep_word(w.head, w.j0 / BN, 2 * (w.it0 + it), 0, drop.keep_nkt, drop.keep_w),
                                      2 * BN * 4, &mbars->full[st]);
                            last[st] = nm + 1;
                        }
                    }
                    if (lead) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, issuer_lane) != 0;   // warp-uniform again
                }
                if (issuer) {
                    if (!ok) fail(bars, status);
                    // never leave the CTA with copies in flight
                    for (int st = 0; st < MSB; ++st)
                        if (last[st]) mbar_wait(&mbars->full[st], ((last[st] - 1) / MSB) & 1, nullptr);
                }
            } else {
                // drawn: thread = key r of the item's key tile, half m of the query rows; the 32
                // decisions of (row i0 + 32m + c, key) as one word, element drawn from its flat index
                // (head*S + i0 + 32m + c)*S + key
                const int r = (mw % 4) * 32 + lane, m = mw / 4;
                for (int k = 0; ok; ++k) {
                    const int item = take_item(bars, k, status, ok);
                    if (item < 0) break;
                    const Item w = item_of(item);
                    const uint64_t key = (uint64_t)(w.j0 + r);
                    const uint64_t step = (uint64_t)S * kDropGolden;
                    for (int it = 0; it < w.n; ++it) {
                        const uint32_t st = nm % MSB;
                        if (nm >= MSB && !(ok = warp_wait(&mbars->empty[st], ((nm / MSB) + 1) & 1, bars, status))) break;
                        const uint64_t i0 = (uint64_t)((w.it0 + it) * BM + 32 * m);
                        uint64_t g = (((uint64_t)w.head * S + i0) * (uint64_t)S + key) * kDropGolden;
                        uint32_t bits = 0u;
#pragma unroll 4
                        for (int b = 0; b < 32; ++b) {
                            bits |= (uint32_t)drop_keep(drop.seed, g, drop.keep_thr) << b;
                            g += step;
                        }
                        mask_w[(st * 2 + m) * BN + r] = bits;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&mbars->full[st]);
                        ++nm;
                    }
                }
            }
        }
    } else if (warp < 4) {
        if (DROP) regs_increase<184>();
        // thread = key row r of the item's key tile (TMEM lane)
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        uint32_t gt = 0;   // query tiles of earlier items
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = take_item(bars, k, status, ok);
            if (item < 0) break;
            const Item w = item_of(item);
            const int head = w.head, j0 = w.j0, it0 = w.it0, n = w.n;
            const int key = j0 + r;
            // K_j row r -> TMEM (bf16 pairs along hd) as the A operand of S^T = K_j Q_i^T; the previous
            // item's S^T MMAs, which read these columns, are done (this warp has waited for them below)
            if ((ok = warp_wait(&bars->kv_full, k & 1, bars, status))) {
#pragma unroll
                for (int sub = 0; sub < C::SUB; ++sub) {
                    uint32_t kw[32];
                    const uint8_t *krow = smem + C::OFF_K + sub * C::KV_SUB + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v4 = *reinterpret_cast<const uint4 *>(krow + ((c ^ (r & 7)) << 4));
                        kw[4 * c + 0] = v4.x;
                        kw[4 * c + 1] = v4.y;
                        kw[4 * c + 2] = v4.z;
                        kw[4 * c + 3] = v4.w;
                    }
                    tmem_st32(tmem + lane_off + C::COL_KT + 32 * sub, kw);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->kt_full);
            }
            for (int it = 0; ok && it < n; ++it) {
                const uint32_t gi = gt + it;
                const int b = gi & 1, st = gi % NSQ;
                const uint32_t ph2 = (gi >> 1) & 1;
                const int i0 = (it0 + it) * BM;
                const float *Ls = ld_s + st * 2 * BM;
                const float *Ds = Ls + BM;
                // dropout: keep bits of (row i0 + c, key) for the 64 columns, drawn ahead by the mask
                // warps (their stages follow the same running tile count)
                uint32_t km[2] = {0u, 0u};
                if (DROP) {
                    const uint32_t mst = gi % MSB;
                    if (!(ok = warp_wait(&mbars->full[mst], (gi / MSB) & 1, bars, status))) break;
                    km[0] = mask_s[(mst * 2) * BN + r];
                    km[1] = mask_s[(mst * 2 + 1) * BN + r];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&mbars->empty[mst]);
                }
                // S^T of this tile: one buffer (phase per tile) or two alternating (phase per pair)
                const uint32_t t_s = tmem + lane_off + C::template col_s<FUSED_DQ>(gi);
                if (!(ok = !TWO_S ? warp_wait(&bars->s_full[0], gi & 1, bars, status)
                                    : warp_wait(&bars->s_full[b], ph2, bars, status)))
                    break;
                tc_fence_after_sync();
                uint32_t sr[64];
                tmem_ld32(t_s, sr);
                tmem_ld32(t_s + 32, sr + 32);
                tmem_wait_ld();
                reg_fence32(sr);
                reg_fence32(sr + 32);
                // p = 2^(s * scale * log2(e) - L * log2(e)) on packed pairs; -L*log2(e) comes from the pre-pass.
                // With dropout the pre-pass adds log2(1 / (1 - p_drop)), so p here is already P / (1 - p_drop):
                // P o C is p where the key is kept and 0 elsewhere, and dS (below) takes D (1 - p_drop) in place of D
                const uint64_t cs2 = f2_pack(scale_log2, scale_log2);
                const bool diag = key > i0;   // some (key > row) pairs in this tile
                uint64_t pp[32];              // P pairs (fp32) kept for dS
                {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(Ls + c);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int cc = c + 2 * h;
                            const float2 a = f2_unpack(ffma2(f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), cs2,
                                                             h == 0 ? f2_pack(l4.x, l4.y) : f2_pack(l4.z, l4.w)));
                            float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
                            if (diag) {
                                if (key > i0 + cc) p0 = 0.0f;
                                if (key > i0 + cc + 1) p1 = 0.0f;
                            }
                            pp[cc / 2] = f2_pack(p0, p1);
                            if (DROP) {
                                const bool k0 = (km[cc / 32] >> (cc % 32)) & 1u;
                                const bool k1 = (km[cc / 32] >> (cc % 32 + 1)) & 1u;
                                pk[cc / 2] = pack_bf16x2(k0 ? p0 : 0.0f, k1 ? p1 : 0.0f);
                            } else {
                                pk[cc / 2] = pack_bf16x2(p0, p1);
                            }
                        }
                    }
                    tmem_st32(t_s, pk);
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full);

                if (!(ok = TWO_DP ? warp_wait(&bars->dp_full[b], ph2, bars, status)
                                  : warp_wait(&bars->dp_full[0], gi & 1, bars, status)))
                    break;
                tc_fence_after_sync();
                // dS buffer b was last read by the dQ^T MMA of tile gi - 2, which the MMA warp issued
                // before this tile's S^T: the S^T commit waited for above tracks it, so the buffer is
                // free.  At hd = 128 the key warps still wait for that MMA's own commit (measured:
                // dropping the wait there made the kernel 4 % slower)
                if (FUSED_DQ && HD == 128 && gi >= 2 && !(ok = warp_wait(&bars->ds_empty[b], ph2 ^ 1, bars, status)))
                    break;
                uint8_t *dsrow = smem + C::OFF_DS + b * C::DS_BYTES + r * 128;
                // dS = P (dP - D) scale on packed pairs; with dropout P (C dP / (1 - p_drop) - D) scale, formed
                // as p (C dP - (1 - p_drop) D) scale from the p / (1 - p_drop) above
                const uint64_t sc2 = f2_pack(scale, scale);
                const uint64_t m1 = DROP ? f2_pack(-drop.keep_frac, -drop.keep_frac) : f2_pack(-1.0f, -1.0f);
                // all 64 dP columns with one tcgen05.wait::ld (each wait waits for every load in flight;
                // one wait instead of two per tile measured 1-5 % faster)
                uint32_t dpa[64];
                const uint32_t t_dp = tmem + lane_off + C::template col_dp<FUSED_DQ>(gi);
                tmem_ld32(t_dp, dpa);
                tmem_ld32(t_dp + 32, dpa + 32);
                tmem_wait_ld();
                reg_fence32(dpa);
                reg_fence32(dpa + 32);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t *dp = dpa + 32 * h;
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c = 32 * h + 2 * e;
                        const float2 d2 = *reinterpret_cast<const float2 *>(Ds + c);
                        float dp0 = __uint_as_float(dp[2 * e]), dp1 = __uint_as_float(dp[2 * e + 1]);
                        if (DROP) {   // the dropout node's backward: C o (dO V^T), its 1 / (1 - p_drop) in p
                            dp0 = (km[c / 32] >> (c % 32)) & 1u ? dp0 : 0.0f;
                            dp1 = (km[c / 32] >> (c % 32 + 1)) & 1u ? dp1 : 0.0f;
                        }
                        const uint64_t t = ffma2(f2_pack(d2.x, d2.y), m1, f2_pack(dp0, dp1));
                        const float2 ds = f2_unpack(fmul2(fmul2(pp[c / 2], sc2), t));
                        pk[e] = pack_bf16x2(ds.x, ds.y);
                    }
                    // dS^T pairs into the dP^T columns already read (A operand of dK += dS^T Q_i)
                    tmem_st16(t_dp + 16 * h, pk);
                    if (FUSED_DQ) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int chunk = 4 * h + v;                   // 16-byte chunk of the 128-byte row
                            uint4 w;
                            w.x = pk[4 * v + 0];
                            w.y = pk[4 * v + 1];
                            w.z = pk[4 * v + 2];
                            w.w = pk[4 * v + 3];
                            *reinterpret_cast<uint4 *>(dsrow + ((chunk ^ (r & 7)) << 4)) = w;
                        }
                    }
                }
                tmem_wait_st();
                if (FUSED_DQ) fence_proxy_async_smem();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->ds_full[b]);
            }
            if (!ok) break;
            // epilogue: dV rows straight from TMEM to global memory once every MMA of the item is done
            if (!(ok = warp_wait(&bars->done, k & 1, bars, status))) break;
            tc_fence_after_sync();
            store_rows_global<HD>(tmem + lane_off + C::COL_DV, dV + ((size_t)head * S + min(key, S - 1)) * HD, key < S);
            gt += n;
        }
    } else if (warp < 8) {
        if (DROP) regs_increase<128>();
        // dQ readout: thread = hd index d (TMEM lane of dQ^T); then the item's dK rows (thread = key)
        const int wq = warp - 4;
        const int d = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint32_t gt = 0;   // query tiles of earlier items
        bool ok = true;
        // at hd = 64 the MMA warp waits for this warp on ds_full before every dQ^T; tile 0 has no
        // predecessor
        if (FUSED_DQ && HD == 64 && d < HD && lane == 0) mbar_arrive(&bars->ds_full[0]);
        for (int k = 0; ok; ++k) {
            const int item = take_item(bars, k, status, ok);
            if (item < 0) break;
            const Item w = item_of(item);
            if (FUSED_DQ && d < HD) {
                for (int it = 0; it < w.n; ++it) {
                    const uint32_t gi = gt + it;
                    // the readout warps stay in step: all leave the loop together if one gives up
                    if (!(ok = named_bar_and(1, HD, warp_wait(&bars->dq_full, gi & 1, bars, status)))) break;
                    tc_fence_after_sync();
                    uint32_t g[64];
                    tmem_ld32(tmem + lane_off + C::COL_DQ, g);
                    tmem_ld32(tmem + lane_off + C::COL_DQ + 32, g + 32);
                    tmem_wait_ld();
                    reg_fence32(g);
                    reg_fence32(g + 32);
                    tc_fence_before_sync();
                    __syncwarp();
                    // dQ^T of tile gi is out of TMEM: the next tile's dQ^T may be issued
                    if (lane == 0) mbar_arrive(HD == 64 ? &bars->ds_full[(gi + 1) & 1] : &bars->dq_empty);
                    const int i0 = (w.it0 + it) * BM;
                    const int rows = min(BM, S - i0);
                    // the staging tile is free once the previous bulk reduce has read it
                    if (d == 0) bulk_wait_group_read0();
                    named_bar_sync(1, HD);
#pragma unroll
                    for (int c = 0; c < BM; ++c) dq_stage[c * HD + d] = __uint_as_float(g[c]);
                    fence_proxy_async_smem();
                    named_bar_sync(1, HD);
                    if (d == 0) {
                        bulk_reduce_add_f32(dq_acc + ((size_t)w.head * S + i0) * HD, dq_stage,
                                            (uint32_t)(rows * HD * 4));
                        bulk_commit_group();
                    }
                }
            }
            if (!ok) break;
            // dK rows (same TMEM lanes as warps 0-3: thread = key) once every MMA of the item is
            // done; then the next item's first dK MMA may overwrite the accumulator
            if (!(ok = warp_wait(&bars->done, k & 1, bars, status))) break;
            tc_fence_after_sync();
            const int key = w.j0 + wq * 32 + lane;
            store_rows_global<HD>(tmem + lane_off + C::COL_DK, dK + ((size_t)w.head * S + min(key, S - 1)) * HD,
                                  key < S);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->dk_read);
            gt += w.n;
        }
        if (FUSED_DQ && d == 0) bulk_wait_group_read0();   // the staging tile is read; the adds complete before the grid does
    }

    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        // this CTA has claimed its last item; the last CTA out returns the counter slot to zero
        __threadfence();
        if (atomicAdd(next_item + 1, 1u) == gridDim.x - 1) {
            next_item[0] = 0u;
            next_item[1] = 0u;
            __threadfence();
        }
    }
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Work-item counters of the persistent key-tile kernel, one slot per launch (see SchedSlots).  The
// last CTA of a launch to finish sets both words back to zero (every CTA has claimed past the end
// of the list by then), so a slot is zero whenever a launch starts -- no memset on the stream,
// and graph replays reuse their slot.  Static memory starts at zero.
__device__ unsigned g_next_item[2 * kSchedSlots];
SchedSlots g_slots;

int next_item_counter(cudaStream_t st, unsigned **ctr)
{
    unsigned slot = 0;
    int rc = sched_slot(st, g_slots, &slot);
    if (rc != XFA_OK) return rc;
    void *base = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&base, g_next_item);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    *ctr = static_cast<unsigned *>(base) + 2 * slot;
    return XFA_OK;
}

template <int HD, bool FUSED_DQ, bool DROP>
int run(const BwdParams &p, cudaStream_t st)
{
    alignas(64) CUtensorMap tk, tv, tq, tdo;
    int rc = encode_tmap_bf16_3d(&tk, p.k, HD, p.S, p.bh, BN);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tv, p.v, HD, p.S, p.bh, BN);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tq, p.q, HD, p.S, p.bh, BM);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tdo, p.dout, HD, p.S, p.bh, BM);
    if (rc != XFA_OK) return rc;
    constexpr int smem = Cfg<HD, DROP>::SMEM;
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    auto kern = tc_bwd_kernel<HD, FUSED_DQ, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    const int nkt = (p.S + BN - 1) / BN;
    const unsigned grid = (unsigned)std::min(nkt * p.bh, device_sm_count());   // persistent: one CTA per SM
    unsigned *ctr = nullptr;
    if ((rc = next_item_counter(st, &ctr)) != XFA_OK) return rc;
    kern<<<grid, DROP ? kThreadsDrop : kThreads, smem, st>>>(tk, tv, tq, tdo, p.Lg, p.D, p.dq_acc, (__nv_bfloat16 *)p.dk,
                                                 (__nv_bfloat16 *)p.dv, p.bh, p.S, p.S_pad, p.scale,
                                                 p.scale * 1.4426950408889634f, p.status, p.drop,
                                                 head_bundle(p.bh, p.S, HD, 2, kHeadBundle), ctr);
    e = cudaGetLastError();
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

}  // namespace

int launch_tc_bwd(const BwdParams &p, cudaStream_t st, bool fused_dq)
{
    if (p.dtype != XFA_BF16) return XFA_ERR_UNSUPPORTED;
    if (p.drop.on && !fused_dq) return XFA_ERR_UNSUPPORTED;   // dropout: fused variant only
    if (p.hd == 128) {
        if (p.drop.on) return run<128, true, true>(p, st);
        return fused_dq ? run<128, true, false>(p, st) : run<128, false, false>(p, st);
    }
    if (p.hd == 64) {
        if (p.drop.on) return run<64, true, true>(p, st);
        return fused_dq ? run<64, true, false>(p, st) : run<64, false, false>(p, st);
    }
    return XFA_ERR_UNSUPPORTED;
}

}  // namespace xfa
