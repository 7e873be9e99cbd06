// Flash-attention forward on the sm_103a tensor cores (bf16 in, fp32 accumulate).
//
// Method: "xtrain docs/13-flash-attention.md", section "什么是 flash-attention":
// for each query row, scan the key/value tiles at or below the diagonal with
// the online softmax (running max m, running sum l, accumulator rescaled by
// exp(m_old - m_new)), finish with out = acc / l and L = m + ln l; tiles wholly
// above the diagonal are never touched.
//
// GB300 design (replaces the page's one-block-per-row SIMT kernel):
//   * persistent CTAs, one per SM; a work item is 256 query rows of one head as two
//     128-row tiles (t = 0, 1), claimed from a per-launch counter (see the kernel);
//   * warp 8 claims items and streams Q and the K and V tiles (128 keys x hd) through
//     a TMA ring with 128-byte swizzle; the ring runs on across items, and the V of
//     each key tile and the K of the next (in the next item after an item's last)
//     land on one barrier, so the MMA thread waits once per key step;
//   * warp 9 (one thread) issues tcgen05.mma: S_t = Q_t K^T into TMEM
//     (128 lanes x 128 fp32 columns) and O_t += P_t V with P_t read straight
//     from TMEM (bf16, packed into the first 64 columns of S_t);
//   * warps 0-3 and 4-7 are the softmax groups of tiles 0 and 1: thread = row,
//     tcgen05.ld of the S row, scaled exp2, row max / sum in registers, P
//     written back with tcgen05.st.  While one group works on its S tile the
//     tensor core runs the other tile's MMAs.
//   * The O rescale is lazy: the reference maximum only moves when a row max
//     exceeds it by more than 2^8 (in exp2 units), so P <= 256 and fp32
//     accumulation is unaffected; when it moves, the warp rescales its O rows
//     in TMEM after the previous P.V has completed (guaranteed by the S-ready
//     commit, which tracks every earlier MMA).
// TMEM map (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+hd) O1 [256+hd, 256+2hd).
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <math_constants.h>

#include "dropout.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace xfa {
namespace {

constexpr int BM = 128;               // query rows per tile (MMA M)
constexpr int BN = 128;               // keys per tile (MMA N of S, K of P.V)
constexpr int kThreads = 320;         // 10 warps
constexpr int kWarpTma = 8, kWarpMma = 9;
// With dropout: 28 warps.  Warps 12-27 (four warpgroups, four warps per SM sub-partition: the draw
// is bound by the integer multiplier, which it shares with the softmax's fp32 arithmetic, and
// more warps keep more draws in flight: 16 warps measured 3-4 % faster than 8, 8 than 4) draw the
// keep bits of every (row, key) of the coming key tiles into shared memory (MS stages per tile),
// one 32-key word per thread, so the softmax warps only read them; warps 10-11 are idle.  An
// 896-thread launch gets 72 registers a thread; they move from the TMA/MMA/idle warpgroup and
// the keep-bit warpgroups to the softmax warpgroups (the counts at the softmax's setmaxnreg).
constexpr int kMaskWarps = 16;
constexpr int kMaskWords = 16 / kMaskWarps;   // 32-key words of a row per keep-bit thread
constexpr int kWarpMask0 = 12;
constexpr int kThreadsDrop = (kWarpMask0 + kMaskWarps) * 32;
constexpr int MS = 2;                 // keep-bit stages per tile
constexpr int kMaskBytes = 2 * MS * 128 * 16;   // [tile][stage][row] x 128 bits
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kHeadBundle = 8;              // heads scheduled together at long S (L2 reuse of K/V)

template <int HD>
struct Cfg {
    static constexpr int SUB = HD / 64;                 // 128-byte column blocks per row
    static constexpr int SUB_BYTES = 128 * 128;         // 128 rows x 128 B
    static constexpr int TILE_BYTES = BM * HD * 2;      // BM == BN
    static constexpr int NS = HD == 128 ? 2 : 3;        // K/V ring depth
    static constexpr int OFF_Q0 = 0;
    static constexpr int OFF_Q1 = TILE_BYTES;
    static constexpr int OFF_K = 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr int OFF_MASK = OFF_BAR + 512;      // keep bits (dropout only)
    template <bool DROP>
    static constexpr int smem() { return OFF_MASK + (DROP ? kMaskBytes : 0) + 1024; }   // + alignment slack
    // TMEM columns of S_t and O_t
    static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * (uint32_t)t; }
    static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + (uint32_t)(HD * t); }
};

struct Bars {
    uint64_t q_full;
    uint64_t q_empty;     // the item's last S MMAs have read Q (tensor-core commit)
    // v_full[s]: the V of the key tile in stage s and the K of the next key tile; k_full[0]: the
    // CTA's first K (k_full[1], k_full[2] are not used); k_empty / v_empty: the stage's K read by
    // its S MMAs / its V read by its P.Vs (tensor-core commits)
    uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
    uint64_t s_full[2];   // S_t ready in TMEM (tensor-core commit)
    uint64_t p_full[2];   // P_t written to TMEM (one arrival per softmax warp)
    uint64_t o_full[2];   // O_t complete (commit after the last P.V)
    uint64_t drain;       // MMA drain at teardown
    uint64_t mask_full[2][MS];   // keep bits of tile t written (one arrival per mask warp)
    uint64_t mask_empty[2][MS];  // read by the softmax group of tile t (one arrival per warp)
    uint64_t item_full[2];   // work-item id posted by the TMA warp
    uint64_t item_empty[2];  // id read by the MMA warp, the eight softmax warps and any keep-bit warps
    int item_id[2];          // the posted ids (-1: no more work)
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void fail(Bars *b, int *status)
{
    b->abort = 1;
    record_status(status, XFA_ERR_TIMEOUT);
}

// All lanes wait; the outcome is made warp-uniform so warp-collective
// tcgen05 instructions after it are never reached by part of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, Bars *b, int *status)
{
    bool ok = mbar_wait_spin(bar, parity, &b->abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) fail(b, status);
    return ok;
}

// The next work item for a consumer warp (MMA or softmax): waits until the TMA warp has posted
// it in ring entry k & 1, reads it and releases the entry (one arrival per warp).  -1: no more
// work, or the wait gave up (then ok is false).
__device__ __forceinline__ int take_item(Bars *b, int k, int *status, bool &ok)
{
    const int e = k & 1;
    if (!(ok = warp_wait(&b->item_full[e], (k >> 1) & 1, b, status))) return -1;
    const int item = *reinterpret_cast<volatile int *>(&b->item_id[e]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&b->item_empty[e]);
    return item;
}

// S = Q K^T: M=128, N=128, K=hd in steps of 16 (K-major, 128-byte swizzle; 64-column blocks SUB_BYTES apart).
template <int HD>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc)
{
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
        const uint32_t off = (ks / 4) * Cfg<HD>::SUB_BYTES + (ks % 4) * 32;
        mma_ss(d_tmem, sdesc_advance(q_desc, off), sdesc_advance(k_desc, off), idesc, ks > 0);
    }
}

// TMEM column (from the start of S_t) of the packed P of keys 16ks .. 16ks + 15.  hd = 128: keys 0-63
// in columns 0-31, keys 64-127 in columns 96-127 (the softmax writes the second half's P from the
// scores it still holds from the maximum pass, over score columns of that half, before it re-reads
// the first half); hd = 64: columns 0-63 in order.
template <int HD>
__host__ __device__ constexpr uint32_t p_col(int ks) { return HD == 128 && ks >= 4 ? 96 + 8 * (ks - 4) : 8 * ks; }

// O += P V: P (bf16) from TMEM, V [keys][hd] as an MN-major B operand; 16 keys = 2048 bytes.
template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, bool accumulate)
{
    constexpr uint32_t idesc = idesc_bf16(BM, HD, false, true);
#pragma unroll
    for (int ks = 0; ks < BN / 16; ++ks)
        mma_ts(o_tmem, p_tmem + p_col<HD>(ks), sdesc_advance(v_desc, ks * 2048), idesc, (accumulate || ks > 0) ? 1u : 0u);
}

// Raw scores of columns 64h..64h+63 of this thread's row of S_t (TMEM lane); on the
// diagonal key tile the keys past the row (column > r) become -inf.
__device__ __forceinline__ void load_scores_half(uint32_t tS, int h, bool diag, int r, uint32_t *sh)
{
    tmem_ld32(tS + 64 * h, sh);
    tmem_ld32(tS + 64 * h + 32, sh + 32);
    tmem_wait_ld();
    reg_fence32(sh);
    reg_fence32(sh + 32);
    if (diag) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (64 * h + c > r) sh[c] = 0xff800000u;   // -inf
    }
}

// DROP: dropout on the probabilities that enter P.V (the row sums l keep every p).
// KEEP (with DROP): the keep bits are read from the cache (DropParams::keep_in) instead of drawn;
// the keep-bit warps then need few registers and the softmax warps get more.
template <int HD, bool DROP, bool KEEP = false>
__global__ void __launch_bounds__(DROP ? kThreadsDrop : kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ O,
                  float *__restrict__ lse, int bh, int S, float scale_log2, int *status, const DropParams drop,
                  int bundle_heads, unsigned *__restrict__ next_item)
{
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Persistent CTAs: the grid has at most one CTA per SM, and each CTA takes work items -- query
    // blocks of 256 rows (two tiles) of one head -- from a shared counter (next_item, zeroed
    // before the launch) until the list is exhausted: greedy scheduling, as the hardware does
    // for a grid of one CTA per item, without the CTA teardown and launch between items.  The
    // list runs heads in bundles of bundle_heads (see head_bundle: at long S the K/V of the
    // heads in flight stay in L2) and, within a bundle, the heaviest (longest) query blocks
    // first.  The TMA warp claims an item and posts its id to the other warps through a
    // two-entry ring; barrier phases and the K/V ring carry over from one item to the next: the
    // next item's Q loads as soon as the current item's last S MMA has read the old one, and its
    // first S MMAs run while the softmax warps still write out the current item's O.
    const int nqb = (S + 2 * BM - 1) / (2 * BM);
    const int n_items = nqb * bh;
    auto item_coords = [&](int item, int &head, int &qb) {
        const int bundle = item / (nqb * bundle_heads);
        const int g = min(bundle_heads, bh - bundle * bundle_heads);   // heads in this bundle
        const int idx = item - bundle * nqb * bundle_heads;
        qb = nqb - 1 - idx / g;
        head = bundle * bundle_heads + idx % g;
    };

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < 3; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], BM / 32);   // one arrival per softmax warp
            mbar_init(&bars->o_full[t], 1);
        }
        mbar_init(&bars->drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->item_full[i], 1);
            // MMA warp + eight softmax warps (+ the keep-bit warps)
            mbar_init(&bars->item_empty[i], 1 + BM / 32 * 2 + (DROP ? kMaskWarps : 0));
        }
        for (int t = 0; t < 2; ++t)
            for (int s = 0; s < MS; ++s) {
                mbar_init(&bars->mask_full[t][s], kMaskWarps);
                mbar_init(&bars->mask_empty[t][s], BM / 32);
            }
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    uint32_t *mask_s = reinterpret_cast<uint32_t *>(smem + C::OFF_MASK);

    // Roles by warpgroup (with dropout every warpgroup first resizes its registers, all four warps
    // together): warps 8-11 the TMA and MMA warps (and two idle ones), 12-19 the keep-bit warps,
    // 0-7 the softmax groups.
    if (warp >= 8 && warp < 12) {
        if (DROP) regs_decrease<56>();
        if (warp == kWarpTma) {
            if (lane == 0) {
                prefetch_tensormap(&tm_q);
                prefetch_tensormap(&tm_k);
                prefetch_tensormap(&tm_v);
                uint32_t g = 0;                       // K/V tiles issued by this CTA
                uint32_t last_v[3] = {0, 0, 0};      // 1 + last tile whose V (and the next K) went to each stage
                int k = 0;                            // items whose Q was issued
                int kc = 0;                           // items claimed, posted in ring entry kc & 1
                bool ok = true;
                // Claim the next work item and post its id to the other warps (-1: no more work).
                auto claim = [&]() -> int {
                    const int e = kc & 1;
                    if (kc >= 2 && !(ok = mbar_wait_spin(&bars->item_empty[e], ((kc >> 1) + 1) & 1, &bars->abort)))
                        return -1;
                    int it = (int)atomicAdd(next_item, 1u);
                    if (it >= n_items) it = -1;
                    *reinterpret_cast<volatile int *>(&bars->item_id[e]) = it;
                    mbar_arrive(&bars->item_full[e]);
                    ++kc;
                    return it;
                };
                // Q of an item: the Q buffers are free once the previous item's last S MMAs have read them.
                auto load_q = [&](int head, int q0, bool t1) {
                    if (k > 0 && !(ok = mbar_wait_spin(&bars->q_empty, (k - 1) & 1, &bars->abort))) return;
                    mbar_arrive_expect_tx(&bars->q_full, (t1 ? 2 : 1) * C::TILE_BYTES);
                    for (int s = 0; s < C::SUB; ++s) {
                        tma_load_3d(smem + C::OFF_Q0 + s * C::SUB_BYTES, &tm_q, &bars->q_full, s * 64, q0, head);
                        if (t1) tma_load_3d(smem + C::OFF_Q1 + s * C::SUB_BYTES, &tm_q, &bars->q_full, s * 64, q0 + BM, head);
                    }
                    ++k;
                };
                // K of the CTA's tile gk (key tile j of `head`) into its stage, completing on `bar`; the stage is
                // free once the S MMAs of tile gk - NS have read it.
                auto load_k = [&](uint32_t gk, int head, int j, uint64_t *bar) {
                    const int st = gk % C::NS;
                    if (gk >= C::NS && !(ok = mbar_wait_spin(&bars->k_empty[st], ((gk / C::NS) + 1) & 1, &bars->abort)))
                        return;
                    for (int s = 0; s < C::SUB; ++s)
                        tma_load_3d(smem + C::OFF_K + st * C::TILE_BYTES + s * C::SUB_BYTES, &tm_k, bar, s * 64, j * BN, head);
                };
                // V of tile g and K of tile g + 1 (the next key tile of the item, or the next item's first)
                // complete on one barrier, v_full[g % NS]: the MMA warp waits once per key step.  The CTA's
                // first K completes on k_full[0].
                bool k0 = false;
                int item = claim();
                if (item >= 0) {
                    int head, qb;
                    item_coords(item, head, qb);
                    int q0 = qb * 2 * BM;
                    bool t1 = q0 + BM < S;
                    int nkv = t1 ? 2 * qb + 2 : 2 * qb + 1;
                    load_q(head, q0, t1);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars->k_full[0], C::TILE_BYTES);
                        load_k(0, head, 0, &bars->k_full[0]);
                        k0 = true;
                    }
                    for (int j = 0; ok;) {
                        const int st = g % C::NS;
                        if (g >= C::NS && !(ok = mbar_wait_spin(&bars->v_empty[st], ((g / C::NS) + 1) & 1, &bars->abort)))
                            break;
                        const bool last = j == nkv - 1;
                        int nitem = item;
                        if (last && (nitem = claim()) < 0 && !ok) break;
                        int nhead = head, nqb = qb, nj = j + 1;
                        if (last && nitem >= 0) {
                            item_coords(nitem, nhead, nqb);
                            nj = 0;
                        }
                        const bool has_next = !last || nitem >= 0;
                        mbar_arrive_expect_tx(&bars->v_full[st], (has_next ? 2 : 1) * C::TILE_BYTES);
                        for (int s = 0; s < C::SUB; ++s)
                            tma_load_3d(smem + C::OFF_V + st * C::TILE_BYTES + s * C::SUB_BYTES, &tm_v, &bars->v_full[st],
                                        s * 64, j * BN, head);
                        last_v[st] = g + 1;
                        if (has_next) load_k(g + 1, nhead, nj, &bars->v_full[st]);
                        ++g;
                        if (!ok || !has_next) break;
                        if (last) {   // on to the next item
                            item = nitem;
                            head = nhead;
                            qb = nqb;
                            q0 = qb * 2 * BM;
                            t1 = q0 + BM < S;
                            nkv = t1 ? 2 * qb + 2 : 2 * qb + 1;
                            load_q(head, q0, t1);
                        }
                        j = nj;
                    }
                }
                if (!ok) fail(bars, status);
                // Never leave the CTA with copies in flight: wait for the last load of Q and of each stage.
                if (k > 0) mbar_wait_spin(&bars->q_full, (k - 1) & 1, nullptr);
                if (k0) mbar_wait_spin(&bars->k_full[0], 0, nullptr);
                for (int st = 0; st < C::NS; ++st)
                    if (last_v[st]) mbar_wait_spin(&bars->v_full[st], ((last_v[st] - 1) / C::NS) & 1, nullptr);
            }
        } else if (warp == kWarpMma) {
            // The whole warp runs the issue loop (converged, so descriptors stay warp-uniform);
            // one elected lane issues the tcgen05 instructions.
            const bool leader = elect_one();
            const uint64_t q_desc[2] = {sdesc_sw128(smem_u32(smem + C::OFF_Q0), 16, 1024),
                                        sdesc_sw128(smem_u32(smem + C::OFF_Q1), 16, 1024)};
            const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::OFF_V), C::SUB_BYTES, 1024);
            uint32_t g = 0;                 // K/V tiles consumed by this CTA
            uint32_t np[2] = {0, 0};        // P phases consumed per tile
            int k = 0;                      // items started
            bool ok = true;
            for (; ok; ++k) {
                const int item = take_item(bars, k, status, ok);
                if (item < 0) break;
                int head, qb;
                item_coords(item, head, qb);
                const int q0 = qb * 2 * BM;
                const bool t1 = q0 + BM < S;
                const int n_t0 = 2 * qb + 1, n_t1 = t1 ? 2 * qb + 2 : 0;
                const int nkv = t1 ? n_t1 : n_t0;
                const int st0 = g % C::NS;
                // the item's first K: the CTA's first on k_full[0], later ones came with the previous V
                ok = warp_wait(&bars->q_full, k & 1, bars, status) && (g > 0 || warp_wait(&bars->k_full[0], 0, bars, status));
                if (!ok) break;
                tc_fence_after_sync();
                if (leader) {
                    // S_0 of both tiles.  Each S buffer last held the previous item's final P, read by
                    // its last P.V issued before: the tensor pipe runs in order.
                    issue_qk<HD>(tmem + C::col_s(0), q_desc[0], sdesc_advance(k_desc, st0 * C::TILE_BYTES));
                    tc_commit(&bars->s_full[0]);
                    if (t1) {
                        issue_qk<HD>(tmem + C::col_s(1), q_desc[1], sdesc_advance(k_desc, st0 * C::TILE_BYTES));
                        tc_commit(&bars->s_full[1]);
                    }
                    tc_commit(&bars->k_empty[st0]);
                    if (nkv == 1) tc_commit(&bars->q_empty);   // no further S of this item reads Q
                }
                __syncwarp();
                for (int j = 0; ok && j < nkv; ++j) {
                    const uint32_t gj = g + j, gn = gj + 1;
                    const int st = gj % C::NS, stn = gn % C::NS;
                    const uint32_t ph = (gj / C::NS) & 1;
                    bool v_ready = false, k_next_ready = false;
                    const int jn = j + 1;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int nt = t == 0 ? n_t0 : n_t1;
                        if (j >= nt) continue;
                        ok = warp_wait(&bars->p_full[t], np[t] & 1, bars, status);
                        ++np[t];
                        // V of this key tile and K of the next arrive together
                        if (ok && !v_ready) ok = v_ready = warp_wait(&bars->v_full[st], ph, bars, status);
                        if (!ok) break;
                        tc_fence_after_sync();
                        if (leader) {
                            issue_pv<HD>(tmem + C::col_o(t), tmem + C::col_s(t), sdesc_advance(v_desc, st * C::TILE_BYTES),
                                         j > 0);
                            if (j == nt - 1) tc_commit(&bars->o_full[t]);
                        }
                        __syncwarp();
                        if (jn < nt) {
                            k_next_ready = true;   // came with this key tile's V
                            tc_fence_after_sync();
                            if (leader) {
                                issue_qk<HD>(tmem + C::col_s(t), q_desc[t], sdesc_advance(k_desc, stn * C::TILE_BYTES));
                                tc_commit(&bars->s_full[t]);
                            }
                            __syncwarp();
                        }
                    }
                    if (!ok) break;
                    if (leader) {
                        if (k_next_ready) tc_commit(&bars->k_empty[stn]);
                        tc_commit(&bars->v_empty[st]);
                        if (jn == nkv - 1) tc_commit(&bars->q_empty);   // the item's last S MMAs are issued
                    }
                    __syncwarp();
                }
                g += nkv;
            }
            if (leader) {
                tc_commit(&bars->drain);
                mbar_wait_spin(&bars->drain, 0, nullptr);
            }
            __syncwarp();
        }
    } else if (warp >= 12) {
        if (DROP) {
            if (KEEP)
                regs_decrease<24>();
            else
                regs_decrease<32>();
            // keep bits (dropout): thread = row r of both tiles, half m of the keys; for every key
            // tile of the item, in the order the softmax groups consume them, the 64 decisions of
            // the row's keys 64m..64m+63 as two 32-bit words, element (row, key) drawn from its flat
            // index (head*S + row)*S + key
            const int mw = warp - kWarpMask0;
            const int r = (mw % 4) * 32 + lane, m = mw / 4;
            uint32_t nm[2] = {0u, 0u};   // stages filled per tile
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = take_item(bars, k, status, ok);
                if (item < 0) break;
                int head, qb;
                item_coords(item, head, qb);
                const int q0 = qb * 2 * BM;
                const bool t1 = q0 + BM < S;
                const int n_t0 = 2 * qb + 1, n_t1 = t1 ? 2 * qb + 2 : 0;
                const int nkv = t1 ? n_t1 : n_t0;
                for (int j = 0; ok && j < nkv; ++j) {
#pragma unroll 1
                    for (int t = 0; t < 2; ++t) {
                        if (j >= (t == 0 ? n_t0 : n_t1)) continue;
                        const uint32_t st = nm[t] % MS;
                        // cached decisions (keep_word: one word per key over this warp's 32 rows), loaded
                        // before the wait for the stage and turned back into one word per row
                        const int wrow = (q0 + t * BM + (mw % 4) * 32) / 32;
                        uint32_t cw[2] = {0u, 0u};
                        if (KEEP) {
                            const uint32_t *src =
                                drop.keep_in + keep_word(head, j, wrow, 32 * kMaskWords * m + lane, drop.keep_nkt, drop.keep_w);
#pragma unroll
                            for (int q = 0; q < kMaskWords; ++q) cw[q] = src[32 * q];
                        }
                        if (nm[t] >= MS &&
                            !(ok = warp_wait(&bars->mask_empty[t][st], ((nm[t] / MS) + 1) & 1, bars, status)))
                            break;
                        uint32_t w[2];
                        if (KEEP) {
#pragma unroll
                            for (int q = 0; q < kMaskWords; ++q) w[q] = warp_transpose_bits32(cw[q], lane);
                        } else {
                            const uint64_t row = (uint64_t)(q0 + t * BM + r);
                            uint64_t g = (((uint64_t)head * S + row) * (uint64_t)S + (uint64_t)(j * BN + 32 * kMaskWords * m)) * kDropGolden;
#pragma unroll
                            for (int q = 0; q < kMaskWords; ++q) {
                                uint32_t bits = 0u;
#pragma unroll
                                for (int b = 0; b < 32; ++b) {
                                    bits |= (uint32_t)drop_keep(drop.seed, g, drop.keep_thr) << b;
                                    g += kDropGolden;
                                }
                                w[q] = bits;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < kMaskWords; ++q) mask_s[((t * MS + st) * BM + r) * 4 + kMaskWords * m + q] = w[q];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->mask_full[t][st]);
                        ++nm[t];
                        if (!KEEP && drop.keep_out) {
                            // the same decisions kept for the backward: one word per key over this
                            // warp's 32 rows (keep_word), 128 contiguous bytes per store
                            uint32_t *dst =
                                drop.keep_out + keep_word(head, j, wrow, 32 * kMaskWords * m + lane, drop.keep_nkt, drop.keep_w);
#pragma unroll
                            for (int q = 0; q < kMaskWords; ++q) dst[32 * q] = warp_transpose_bits32(w[q], lane);
                        }
                    }
                }
            }
        }
    } else {
        // 896 threads x 72 registers: per lane of a warpgroup 2 x 152 + 56 + 4 x 32 = 488 (drawing),
        // 2 x 176 + 56 + 4 x 24 = 504 (reading the cache), within 7 x 72 = 504
        if (DROP) {
            if (KEEP)
                regs_increase<176>();
            else
                regs_increase<152>();
        }
        // softmax group of tile t; thread = query row
        const int t = warp / 4, wq = warp % 4;
        const int r = wq * 32 + lane;               // row within the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::col_s(t);
        const uint32_t tO = tmem + lane_off + C::col_o(t);
        uint32_t ns = 0, no = 0;                    // S and O phases of this tile consumed
        uint32_t nmask = 0;                         // keep-bit stages consumed (dropout)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = take_item(bars, k, status, ok);
            if (item < 0) break;
            int head, qb;
            item_coords(item, head, qb);
            const int q0 = qb * 2 * BM;
            const bool t1 = q0 + BM < S;
            if (t == 1 && !t1) continue;                // this item has no second tile
            const int n_mine = t == 0 ? 2 * qb + 1 : 2 * qb + 2;
            const int row = q0 + t * BM + r;
            const int diag = 2 * qb + t;                // key tile that holds this tile's diagonal
            float m = -CUDART_INF_F, l = 0.0f;
            for (int j = 0; j < n_mine; ++j) {
                if (!(ok = warp_wait(&bars->s_full[t], ns & 1, bars, status))) break;
                ++ns;
                tc_fence_after_sync();
                // pass 1: row maximum, the scores read from TMEM in two 64-column halves (so only half
                // a row is held in registers); the diagonal tile masks keys past the row.  4 independent
                // chains of 3-input maxima.
                const bool on_diag = j == diag;
                float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
                // hd = 128: the second half's scores (s1) stay in registers for the exponential pass
                uint32_t s0[64], s1[64];
                if (HD == 64 && !on_diag) {
                    // no masked keys: TMEM loads that reduce while loading (max of 32 columns each).
                    // At hd = 64, where the softmax sets the pace, this is 4 % faster; at hd = 128 it
                    // measured no better than the plain loads, which are kept there.
#pragma unroll
                    for (int q = 0; q < 4; ++q) mx4[q] = tmem_ld32_max(tS + 32 * q);
                    tmem_wait_ld();
                    reg_fence_f4(mx4[0], mx4[1], mx4[2], mx4[3]);
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t *sh = h == 0 ? s0 : s1;
                        load_scores_half(tS, h, on_diag, r, sh);
#pragma unroll
                        for (int c = 0; c < 64; c += 8)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                mx4[e] = fmax3(mx4[e], __uint_as_float(sh[c + 2 * e]), __uint_as_float(sh[c + 2 * e + 1]));
                    }
                }
                const float mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
                const float m_new = fmaxf(m, mx * scale_log2);   // scale > 0: max commutes with the scaling
                const bool need = m_new > m + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = ex2_approx(m - m_new);   // 0 on the first tile
                    l *= alpha;
                    if (j > 0) {
#pragma unroll 1
                        for (int c = 0; c < HD; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(tO + c, o);
                            tmem_wait_ld();
                            reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c, o);
                        }
                        tmem_wait_st();
                    }
                    m = m_new;
                }
                // dropout: this row's keep bits of key tile j, drawn ahead by the mask warps
                uint32_t kb[4] = {0u, 0u, 0u, 0u};
                if (DROP) {
                    const uint32_t st = nmask % MS;
                    if (!(ok = warp_wait(&bars->mask_full[t][st], (nmask / MS) & 1, bars, status))) break;
                    const uint4 v = *reinterpret_cast<const uint4 *>(mask_s + ((t * MS + st) * BM + r) * 4);
                    kb[0] = v.x;
                    kb[1] = v.y;
                    kb[2] = v.z;
                    kb[3] = v.w;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->mask_empty[t][st]);
                    ++nmask;
                }
                // p = 2^(s * scale * log2(e) - m): packed FFMA pairs + ex2; 4 packed partial row sums
                const uint64_t c2 = f2_pack(scale_log2, scale_log2);
                const uint64_t nm2 = f2_pack(-m, -m);
                uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};
                // pass 2: the exponentials, half a row at a time.  hd = 128: the second half first, from
                // the registers of the maximum pass (its P over its own score columns 96-127), then the
                // first half read again (P over columns 0-31); hd = 64: both halves read again, in order.
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = HD == 128 ? 1 - hh : hh;
                    uint32_t *sh = HD == 128 && h == 1 ? s1 : s0;
                    if (!(HD == 128 && h == 1)) load_scores_half(tS, h, on_diag, r, sh);
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c = 64 * h + 2 * e;
                        const float2 a = f2_unpack(ffma2(f2_pack(__uint_as_float(sh[2 * e]), __uint_as_float(sh[2 * e + 1])), c2, nm2));
                        const float p0 = ex2_approx(a.x);
                        const float p1 = ex2_approx(a.y);
                        l2[e & 3] = fadd2(l2[e & 3], f2_pack(p0, p1));
                        if (DROP) {
                            // keys j*BN + c, c + 1 of this row; the factor 1 / (1 - p_drop) is applied to O once, at the end
                            const float d0 = (kb[c >> 5] >> (c & 31)) & 1u ? p0 : 0.0f;
                            const float d1 = (kb[c >> 5] >> ((c + 1) & 31)) & 1u ? p1 : 0.0f;
                            pk[e] = pack_bf16x2(d0, d1);
                        } else {
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                    }
                    tmem_st32(tS + p_col<HD>(4 * h), pk);
                }
                {
                    const float2 a = f2_unpack(fadd2(fadd2(l2[0], l2[1]), fadd2(l2[2], l2[3])));
                    l += a.x + a.y;
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[t]);
            }
            if (!ok) break;
            if (!(ok = warp_wait(&bars->o_full[t], no & 1, bars, status))) break;
            ++no;
            {
                tc_fence_after_sync();
                const float inv_l = (DROP ? drop.inv_keep : 1.0f) / l;
                __nv_bfloat16 *orow = O + ((size_t)head * S + row) * HD;
#pragma unroll 1
                for (int c = 0; c < HD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
                    tmem_wait_ld();
                    reg_fence32(o);
                    if (row < S) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
                            dst[v] = w;
                        }
                    }
                }
                if (row < S) lse[(size_t)head * S + row] = (m + __log2f(l)) * kLn2;
            }
        }
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
        tmem_dealloc(tmem, 512);
    }
}

// Work-item counters of the persistent forward, one slot per launch (see SchedSlots).  The
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

template <int HD, bool DROP, bool KEEP = false>
int run(const FwdParams &p, cudaStream_t st)
{
    alignas(64) CUtensorMap tq, tk, tv;
    int rc = encode_tmap_bf16_3d(&tq, p.q, HD, p.S, p.bh, BM);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tk, p.k, HD, p.S, p.bh, BN);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tv, p.v, HD, p.S, p.bh, BN);
    if (rc != XFA_OK) return rc;
    constexpr int smem = Cfg<HD>::template smem<DROP>();
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    auto kern = tc_fwd_kernel<HD, DROP, KEEP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    const int nqb = (p.S + 2 * BM - 1) / (2 * BM);
    const unsigned grid = (unsigned)std::min(nqb * p.bh, device_sm_count());   // persistent: one CTA per SM
    unsigned *ctr = nullptr;
    if ((rc = next_item_counter(st, &ctr)) != XFA_OK) return rc;
    kern<<<grid, DROP ? kThreadsDrop : kThreads, smem, st>>>(tq, tk, tv, (__nv_bfloat16 *)p.out, p.lse, p.bh, p.S,
                                                 p.scale * 1.4426950408889634f, p.status, p.drop,
                                                 head_bundle(p.bh, p.S, HD, 2, kHeadBundle), ctr);
    e = cudaGetLastError();
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

}  // namespace

int launch_tc_fwd(const FwdParams &p, cudaStream_t st)
{
    if (p.dtype != XFA_BF16) return XFA_ERR_UNSUPPORTED;
    if (p.hd == 128) {
        if (p.drop.on) return p.drop.keep_in ? run<128, true, true>(p, st) : run<128, true>(p, st);
        return run<128, false>(p, st);
    }
    if (p.hd == 64) {
        if (p.drop.on) return p.drop.keep_in ? run<64, true, true>(p, st) : run<64, true>(p, st);
        return run<64, false>(p, st);
    }
    return XFA_ERR_UNSUPPORTED;
}

}  // namespace xfa
