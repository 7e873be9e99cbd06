// Flash-attention backward for fp32 tensors on the sm_103a tensor cores (3xTF32).
//
// Method: "xtrain docs/13-flash-attention.md", section "什么是 flash-attention" (backward):
// P is recomputed from the saved L (p = exp(s - L_i)), dP = dO V^T, dS = P o (dP - D_i) * scale
// with D_i = dO_i . O_i from the pre-pass, then dV = P^T dO, dK = dS^T Q, dQ = dS K.  Every
// contraction is formed by the split of tf32x3.cuh (three kind::tf32 MMAs per product).
//
// GB300 design: two kernels, neither with atomics (the result is bit-reproducible):
//   * tf_bwd_kv_kernel: a CTA owns 128 keys of one head (MMA M).  K and V are split once into
//     TMEM as A operands; dK and dV accumulate in TMEM over every 32-row query tile at or below
//     the diagonal.  Per tile: S^T = K Q^T and dP^T = V dO^T (N = 32), the compute warps
//     (thread = key) form P^T and dS^T and write their hi / lo parts back into TMEM as the A
//     operands of dV += P^T dO and dK += dS^T Q.
//   * tf_bwd_q_kernel: a CTA owns 128 query rows.  Q and dO are split into TMEM; per 32-key
//     tile S = Q K^T, dP = dO V^T, the compute warps (thread = row) form dS, and dQ += dS K.
// Warps 4-7 of each kernel (split group) read the streamed operands from global memory and
// write them as K-major 128-byte-swizzled hi / lo tiles, transposing where the contraction
// runs over rows (Q^T and dO^T for dK and dV, K^T for dQ), so that every shared-memory
// operand is K-major.
#include <math_constants.h>

#include "dropout.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tf32x3.cuh"

namespace xfa {
namespace {

constexpr int BT = 128;               // rows a CTA owns (MMA M)
constexpr int BS = 32;                // rows of a streamed tile (MMA N of S^T, dP^T; K of dV, dK, dQ)
constexpr int kThreads = 288;         // 9 warps
constexpr int kWarpSplit = 4, kWarpMma = 8;
constexpr int NS = 3;                 // depth of the streamed-tile ring

struct Bars {
    uint64_t own_ready;               // the CTA's own rows split into TMEM (one arrival per split warp)
    uint64_t full[NS];                // streamed stage written (one arrival per split warp)
    uint64_t empty[NS];               // stage released (tensor-core commit)
    uint64_t s_full;                  // the two score-shaped products of a tile are in TMEM
    uint64_t p_full;                  // the compute warps wrote their A operands (one arrival per warp)
    uint64_t acc_done;                // every MMA of the CTA complete
    uint64_t drain;
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

__device__ __forceinline__ void init_bars(Bars *bars)
{
    mbar_init(&bars->own_ready, 4);
    for (int s = 0; s < NS; ++s) {
        mbar_init(&bars->full[s], 4);
        mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
}

// D (+)= A B^T with M = 128, A = a_hi / a_lo in TMEM (K columns), B = b_hi / b_lo K-major in
// shared memory; K = 8 * KS, where step ks sits in 128-byte block ks / 4 (`blk` bytes apart).
template <int N, int KS>
__device__ __forceinline__ void mma3(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                     uint32_t blk, bool accumulate)
{
    constexpr uint32_t idesc = idesc_tf32(BT, N);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const uint32_t off = (ks / 4) * blk + (ks % 4) * 32;
        mma_ts_tf32(d, a_hi + 8 * ks, sdesc_advance(b_hi, off), idesc, (accumulate || ks > 0) ? 1u : 0u);
        mma_ts_tf32(d, a_hi + 8 * ks, sdesc_advance(b_lo, off), idesc, 1u);
        mma_ts_tf32(d, a_lo + 8 * ks, sdesc_advance(b_hi, off), idesc, 1u);
    }
}

// One streamed [BS rows x HD] fp32 tile from global memory (rows past S read as zero) into a
// K-major hi / lo pair (`khi`, `klo`: HD / 32 blocks of BS rows x 128 B) and, when T, also its
// transpose (`thi`, `tlo`: HD rows x 128 B, the BS rows contiguous).  128 threads (warp w of the
// group, lane).  A warp takes 16 consecutive rows x 2 adjacent 16-byte columns: each row's 32
// bytes are one sector of the global read, and with the 128-byte swizzle both the 16-byte
// K-major stores and the 4-byte transposed stores of a warp fall in distinct banks.
template <int HD, bool T>
__device__ __forceinline__ void split_tile(const float *src, int row0, int S, int w, int lane, uint8_t *khi,
                                           uint8_t *klo, uint8_t *thi, uint8_t *tlo)
{
    constexpr int F4 = HD / 4;
    constexpr uint32_t BLK = BS * 128;
#pragma unroll
    for (int it = 0; it < BS * F4 / 128; ++it) {
        const int combo = it * 4 + w;                 // (16-row block, column pair)
        const int r = (combo / (F4 / 2)) * 16 + (lane & 15);
        const int c4 = (combo % (F4 / 2)) * 2 + (lane >> 4);
        const bool valid = row0 + r < S;
        const float4 x = ldg4_or_zero(src + (size_t)(valid ? row0 + r : 0) * HD + 4 * c4, valid);
        float4 hi, lo;
        split4(x, hi, lo);
        const uint32_t off = (c4 / 8) * BLK + sw128(r, c4 % 8);
        *reinterpret_cast<float4 *>(khi + off) = hi;
        *reinterpret_cast<float4 *>(klo + off) = lo;
        if (T) {
            const float hs[4] = {hi.x, hi.y, hi.z, hi.w}, ls[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t toff = sw128_word(4 * c4 + e, r);
                *reinterpret_cast<float *>(thi + toff) = hs[e];
                *reinterpret_cast<float *>(tlo + toff) = ls[e];
            }
        }
    }
}

// Store one TMEM row of HD fp32 accumulator columns (thread = lane) to dst when valid.
template <int HD>
__device__ __forceinline__ void tmem_row_to_global(uint32_t t, float *dst, bool valid)
{
#pragma unroll 1
    for (int c = 0; c < HD; c += 32) {
        uint32_t v[32];
        tmem_ld32(t + c, v);
        tmem_wait_ld();
        reg_fence32(v);
        if (valid) {
            float4 *d4 = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                d4[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                    __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
    }
}

// ---------------------------------------------------------------- dK, dV by key tiles

template <int HD>
struct KvCfg {
    static constexpr int MAT = BS * HD * 4;   // one streamed operand tile
    // stage: Q, dO (K-major, B of S^T / dP^T) and Q^T, dO^T (B of dK / dV), each as hi, lo
    static constexpr int OFF_QHI = 0, OFF_QLO = MAT, OFF_OHI = 2 * MAT, OFF_OLO = 3 * MAT;
    static constexpr int OFF_QTHI = 4 * MAT, OFF_QTLO = 5 * MAT, OFF_OTHI = 6 * MAT, OFF_OTLO = 7 * MAT;
    static constexpr int STAGE = 8 * MAT;
    static constexpr int OFF_SCR = NS * STAGE;          // per compute warp: 32 Lg + 32 D
    static constexpr int OFF_BAR = OFF_SCR + 4 * 64 * 4;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static constexpr uint32_t KHI = 0, KLO = HD, VHI = 2 * HD, VLO = 3 * HD;
    static constexpr uint32_t ST = 4 * HD, PLO = ST + BS, DPT = ST + 2 * BS, DSLO = ST + 3 * BS;
    static constexpr uint32_t DV = ST + 4 * BS, DK = DV + HD;
    static_assert(DK + HD <= 512, "TMEM columns");
};

// DROP: dropout's backward (dV takes P o C, dS takes C o dP; see dropout.cuh for C).
template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    tf_bwd_kv_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                     const float *__restrict__ dO, const float *__restrict__ Dg, const float *__restrict__ Lg,
                     float *__restrict__ dK, float *__restrict__ dV, int bh, int S, int S_pad, float scale,
                     float scale_log2, int *status, const DropParams drop)
{
    using C = KvCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int kt = (int)blockIdx.x / bh;             // longest key tiles (most query rows) first
    const int head = (int)blockIdx.x % bh;
    const int k0 = kt * BT;
    const int nq = (S + BS - 1) / BS - k0 / BS;       // query tiles at or below the diagonal
    const size_t hoff = (size_t)head * S * HD;

    if (threadIdx.x == 0) init_bars(bars);
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp >= kWarpSplit && warp < kWarpMma) {
        const int w = warp - kWarpSplit;
        const int tid = threadIdx.x - kWarpSplit * 32;
        {
            const int key = k0 + tid;
            const bool valid = key < S;
            const size_t roff = hoff + (size_t)min(key, S - 1) * HD;
            const uint32_t t = tmem + ((uint32_t)(w * 32) << 16);
            row_to_tmem_split<HD>(K + roff, valid, t + C::KHI, t + C::KLO);
            row_to_tmem_split<HD>(V + roff, valid, t + C::VHI, t + C::VLO);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->own_ready);
        }
        for (int i = 0; i < nq; ++i) {
            const int st = i % NS;
            if (i >= NS && !warp_wait(&bars->empty[st], ((i / NS) + 1) & 1, bars, status)) break;
            uint8_t *g = smem + st * C::STAGE;
            const int q0 = k0 + i * BS;
            split_tile<HD, true>(Q + hoff, q0, S, w, lane, g + C::OFF_QHI, g + C::OFF_QLO, g + C::OFF_QTHI, g + C::OFF_QTLO);
            split_tile<HD, true>(dO + hoff, q0, S, w, lane, g + C::OFF_OHI, g + C::OFF_OLO, g + C::OFF_OTHI,
                                 g + C::OFF_OTLO);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[st]);
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint32_t base = smem_u32(smem);
        auto desc = [&](int st, int off) { return sdesc_sw128(base + st * C::STAGE + off, 16, 1024); };
        constexpr uint32_t BLK = BS * 128;
        bool ok = warp_wait(&bars->own_ready, 0, bars, status) && warp_wait(&bars->full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) {
                mma3<BS, HD / 8>(tmem + C::ST, tmem + C::KHI, tmem + C::KLO, desc(0, C::OFF_QHI), desc(0, C::OFF_QLO),
                                 BLK, false);
                mma3<BS, HD / 8>(tmem + C::DPT, tmem + C::VHI, tmem + C::VLO, desc(0, C::OFF_OHI),
                                 desc(0, C::OFF_OLO), BLK, false);
                tc_commit(&bars->s_full);
            }
            __syncwarp();
        }
        for (int i = 0; ok && i < nq; ++i) {
            if (!(ok = warp_wait(&bars->p_full, i & 1, bars, status))) break;
            tc_fence_after_sync();
            const int st = i % NS;
            if (leader) {
                // dV += P^T dO, dK += dS^T Q: K = the 32 query rows (one 128-byte block)
                mma3<HD, BS / 8>(tmem + C::DV, tmem + C::ST, tmem + C::PLO, desc(st, C::OFF_OTHI),
                                 desc(st, C::OFF_OTLO), 0, i > 0);
                mma3<HD, BS / 8>(tmem + C::DK, tmem + C::DPT, tmem + C::DSLO, desc(st, C::OFF_QTHI),
                                 desc(st, C::OFF_QTLO), 0, i > 0);
                tc_commit(&bars->empty[st]);
                if (i == nq - 1) tc_commit(&bars->acc_done);
            }
            __syncwarp();
            if (i + 1 < nq) {
                const int sn = (i + 1) % NS;
                if (!(ok = warp_wait(&bars->full[sn], ((i + 1) / NS) & 1, bars, status))) break;
                tc_fence_after_sync();
                if (leader) {
                    // overwrite the P^T / dS^T columns the dV / dK MMAs above read: in order
                    mma3<BS, HD / 8>(tmem + C::ST, tmem + C::KHI, tmem + C::KLO, desc(sn, C::OFF_QHI),
                                     desc(sn, C::OFF_QLO), BLK, false);
                    mma3<BS, HD / 8>(tmem + C::DPT, tmem + C::VHI, tmem + C::VLO, desc(sn, C::OFF_OHI),
                                     desc(sn, C::OFF_OLO), BLK, false);
                    tc_commit(&bars->s_full);
                }
                __syncwarp();
            }
        }
        if (leader) {
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0, nullptr);
        }
        __syncwarp();
    } else {
        // compute warps, thread = key (TMEM lane)
        const int key = k0 + warp * 32 + lane;
        const uint32_t t = tmem + ((uint32_t)(warp * 32) << 16);
        float *scr = reinterpret_cast<float *>(smem + C::OFF_SCR) + warp * 64;
        const float *lg_h = Lg + (size_t)head * S_pad, *d_h = Dg + (size_t)head * S_pad;
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
            const int q0 = k0 + i * BS;
            __syncwarp();
            scr[lane] = lg_h[q0 + lane];          // rows past S: Lg = -inf, so p = 0
            scr[32 + lane] = d_h[q0 + lane];
            __syncwarp();
            if (!(ok = warp_wait(&bars->s_full, i & 1, bars, status))) break;
            tc_fence_after_sync();
            uint32_t s[32], dp[32];
            tmem_ld32(t + C::ST, s);
            tmem_ld32(t + C::DPT, dp);
            tmem_wait_ld();
            reg_fence32(s);
            reg_fence32(dp);
            uint32_t p_hi[32], p_lo[32];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 lg = reinterpret_cast<const float4 *>(scr)[c4];
                const float4 dd = reinterpret_cast<const float4 *>(scr + 32)[c4];
                const float lgs[4] = {lg.x, lg.y, lg.z, lg.w}, dds[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * c4 + e;
                    const float p = key <= q0 + c ? ex2_approx(fmaf(__uint_as_float(s[c]), scale_log2, lgs[e])) : 0.0f;
                    float dpc = __uint_as_float(dp[c]), pv = p;
                    if (DROP) {
                        // element (q0 + c, key): flat index (head*S + q0 + c)*S + key
                        const uint64_t g =
                            (((uint64_t)head * S + (uint64_t)(q0 + c)) * (uint64_t)S + (uint64_t)key) * kDropGolden;
                        const bool keep = drop_keep(drop.seed, g, drop.keep_thr);
                        pv = keep ? p * drop.inv_keep : 0.0f;
                        dpc = keep ? dpc * drop.inv_keep : 0.0f;
                    }
                    const float ds = p * (dpc - dds[e]) * scale;
                    split_tf32(pv, p_hi[c], p_lo[c]);
                    split_tf32(ds, s[c], dp[c]);   // s, dp now hold dS^T hi / lo
                }
            }
            tmem_st32(t + C::ST, p_hi);
            tmem_st32(t + C::PLO, p_lo);
            tmem_st32(t + C::DPT, s);
            tmem_st32(t + C::DSLO, dp);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);
        }
        if (ok && nq > 0 && warp_wait(&bars->acc_done, 0, bars, status)) {
            tc_fence_after_sync();
            const size_t roff = (size_t)head * S * HD + (size_t)min(key, S - 1) * HD;
            tmem_row_to_global<HD>(t + C::DV, dV + roff, key < S);
            tmem_row_to_global<HD>(t + C::DK, dK + roff, key < S);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dQ by query tiles

template <int HD>
struct QCfg {
    static constexpr int MAT = BS * HD * 4;
    // stage: K, V (K-major, B of S / dP) and K^T (B of dQ), each as hi, lo
    static constexpr int OFF_KHI = 0, OFF_KLO = MAT, OFF_VHI = 2 * MAT, OFF_VLO = 3 * MAT;
    static constexpr int OFF_KTHI = 4 * MAT, OFF_KTLO = 5 * MAT;
    static constexpr int STAGE = 6 * MAT;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static constexpr uint32_t QHI = 0, QLO = HD, OHI = 2 * HD, OLO = 3 * HD;
    static constexpr uint32_t SC = 4 * HD, DP = SC + BS, DSLO = SC + 2 * BS, DQ = SC + 3 * BS;
    static_assert(DQ + HD <= 512, "TMEM columns");
};

template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    tf_bwd_q_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                    const float *__restrict__ dO, const float *__restrict__ Dg, const float *__restrict__ Lg,
                    float *__restrict__ dQ, int bh, int S, int S_pad, float scale, float scale_log2, int *status,
                    const DropParams drop)
{
    using C = QCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int nqt = (S + BT - 1) / BT;
    const int qt = nqt - 1 - (int)blockIdx.x / bh;   // longest query tiles first
    const int head = (int)blockIdx.x % bh;
    const int q0 = qt * BT;
    const int nk = (min(S, q0 + BT) + BS - 1) / BS;   // key tiles at or below the diagonal
    const size_t hoff = (size_t)head * S * HD;

    if (threadIdx.x == 0) init_bars(bars);
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp >= kWarpSplit && warp < kWarpMma) {
        const int w = warp - kWarpSplit;
        const int tid = threadIdx.x - kWarpSplit * 32;
        {
            const int row = q0 + tid;
            const bool valid = row < S;
            const size_t roff = hoff + (size_t)min(row, S - 1) * HD;
            const uint32_t t = tmem + ((uint32_t)(w * 32) << 16);
            row_to_tmem_split<HD>(Q + roff, valid, t + C::QHI, t + C::QLO);
            row_to_tmem_split<HD>(dO + roff, valid, t + C::OHI, t + C::OLO);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->own_ready);
        }
        for (int j = 0; j < nk; ++j) {
            const int st = j % NS;
            if (j >= NS && !warp_wait(&bars->empty[st], ((j / NS) + 1) & 1, bars, status)) break;
            uint8_t *g = smem + st * C::STAGE;
            split_tile<HD, true>(K + hoff, j * BS, S, w, lane, g + C::OFF_KHI, g + C::OFF_KLO, g + C::OFF_KTHI,
                                 g + C::OFF_KTLO);
            split_tile<HD, false>(V + hoff, j * BS, S, w, lane, g + C::OFF_VHI, g + C::OFF_VLO, nullptr, nullptr);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[st]);
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint32_t base = smem_u32(smem);
        auto desc = [&](int st, int off) { return sdesc_sw128(base + st * C::STAGE + off, 16, 1024); };
        constexpr uint32_t BLK = BS * 128;
        bool ok = warp_wait(&bars->own_ready, 0, bars, status) && warp_wait(&bars->full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) {
                mma3<BS, HD / 8>(tmem + C::SC, tmem + C::QHI, tmem + C::QLO, desc(0, C::OFF_KHI), desc(0, C::OFF_KLO),
                                 BLK, false);
                mma3<BS, HD / 8>(tmem + C::DP, tmem + C::OHI, tmem + C::OLO, desc(0, C::OFF_VHI), desc(0, C::OFF_VLO),
                                 BLK, false);
                tc_commit(&bars->s_full);
            }
            __syncwarp();
        }
        for (int j = 0; ok && j < nk; ++j) {
            if (!(ok = warp_wait(&bars->p_full, j & 1, bars, status))) break;
            tc_fence_after_sync();
            const int st = j % NS;
            if (leader) {
                // dQ += dS K: A = dS_hi (over dP) / dS_lo, B = K^T (K = the 32 keys)
                mma3<HD, BS / 8>(tmem + C::DQ, tmem + C::DP, tmem + C::DSLO, desc(st, C::OFF_KTHI),
                                 desc(st, C::OFF_KTLO), 0, j > 0);
                tc_commit(&bars->empty[st]);
                if (j == nk - 1) tc_commit(&bars->acc_done);
            }
            __syncwarp();
            if (j + 1 < nk) {
                const int sn = (j + 1) % NS;
                if (!(ok = warp_wait(&bars->full[sn], ((j + 1) / NS) & 1, bars, status))) break;
                tc_fence_after_sync();
                if (leader) {
                    mma3<BS, HD / 8>(tmem + C::SC, tmem + C::QHI, tmem + C::QLO, desc(sn, C::OFF_KHI),
                                     desc(sn, C::OFF_KLO), BLK, false);
                    mma3<BS, HD / 8>(tmem + C::DP, tmem + C::OHI, tmem + C::OLO, desc(sn, C::OFF_VHI),
                                     desc(sn, C::OFF_VLO), BLK, false);
                    tc_commit(&bars->s_full);
                }
                __syncwarp();
            }
        }
        if (leader) {
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0, nullptr);
        }
        __syncwarp();
    } else {
        // compute warps, thread = query row (TMEM lane)
        const int row = q0 + warp * 32 + lane;
        const uint32_t t = tmem + ((uint32_t)(warp * 32) << 16);
        const float lg = Lg[(size_t)head * S_pad + row];   // rows past S: -inf, so p = 0
        const float dd = Dg[(size_t)head * S_pad + row];
        bool ok = true;
        for (int j = 0; j < nk; ++j) {
            if (!(ok = warp_wait(&bars->s_full, j & 1, bars, status))) break;
            tc_fence_after_sync();
            uint32_t s[32], dp[32];
            tmem_ld32(t + C::SC, s);
            tmem_ld32(t + C::DP, dp);
            tmem_wait_ld();
            reg_fence32(s);
            reg_fence32(dp);
            const int kmax = row - j * BS;   // columns past this are keys after the row
            // dropout: element (row, key) has flat index (head*S + row)*S + key
            uint64_t drop_g =
                DROP ? (((uint64_t)head * S + (uint64_t)row) * (uint64_t)S + (uint64_t)(j * BS)) * kDropGolden : 0ull;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p = c <= kmax ? ex2_approx(fmaf(__uint_as_float(s[c]), scale_log2, lg)) : 0.0f;
                float dpc = __uint_as_float(dp[c]);
                if (DROP) {
                    dpc = drop_keep(drop.seed, drop_g, drop.keep_thr) ? dpc * drop.inv_keep : 0.0f;
                    drop_g += kDropGolden;
                }
                split_tf32(p * (dpc - dd) * scale, s[c], dp[c]);   // dS hi / lo
            }
            tmem_st32(t + C::DP, s);
            tmem_st32(t + C::DSLO, dp);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);
        }
        if (ok && warp_wait(&bars->acc_done, 0, bars, status)) {
            tc_fence_after_sync();
            tmem_row_to_global<HD>(t + C::DQ, dQ + hoff + (size_t)min(row, S - 1) * HD, row < S);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <typename Kern>
int set_smem(Kern kern, int bytes)
{
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

template <int HD, bool DROP>
int run(const BwdParams &p, cudaStream_t st)
{
    static_assert(KvCfg<HD>::SMEM <= 227 * 1024 && QCfg<HD>::SMEM <= 227 * 1024, "shared memory per CTA");
    const float scale_log2 = p.scale * 1.4426950408889634f;
    const unsigned grid = (unsigned)(((p.S + BT - 1) / BT) * p.bh);
    auto kv = tf_bwd_kv_kernel<HD, DROP>;
    auto qk = tf_bwd_q_kernel<HD, DROP>;
    int rc = set_smem(kv, KvCfg<HD>::SMEM);
    if (rc == XFA_OK) rc = set_smem(qk, QCfg<HD>::SMEM);
    if (rc != XFA_OK) return rc;
    const float *q = (const float *)p.q, *k = (const float *)p.k, *v = (const float *)p.v, *dout = (const float *)p.dout;
    kv<<<grid, kThreads, KvCfg<HD>::SMEM, st>>>(q, k, v, dout, p.D, p.Lg, (float *)p.dk, (float *)p.dv, p.bh, p.S,
                                                 p.S_pad, p.scale, scale_log2, p.status, p.drop);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    qk<<<grid, kThreads, QCfg<HD>::SMEM, st>>>(q, k, v, dout, p.D, p.Lg, (float *)p.dq, p.bh, p.S, p.S_pad, p.scale,
                                                scale_log2, p.status, p.drop);
    e = cudaGetLastError();
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

}  // namespace

int launch_tf_bwd(const BwdParams &p, cudaStream_t st)
{
    if (p.dtype != XFA_F32) return XFA_ERR_UNSUPPORTED;
    if (p.hd == 64) return p.drop.on ? run<64, true>(p, st) : run<64, false>(p, st);
    if (p.hd == 32) return p.drop.on ? run<32, true>(p, st) : run<32, false>(p, st);
    return XFA_ERR_UNSUPPORTED;
}

}  // namespace xfa
