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
constexpr int NS = 3;                 // most stages of a streamed-tile ring

struct Bars {
    uint64_t own_ready;               // the CTA's own rows split into TMEM (one arrival per split warp)
    uint64_t full[NS];                // streamed stage written (one arrival per split warp)
    uint64_t empty[NS];               // stage released (tensor-core commit)
    uint64_t s_full[2];               // buffer b: the two score-shaped products of a tile are in TMEM
    uint64_t p_full[2];               // buffer b: the compute warps wrote their A operands (one per warp)
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
    for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->s_full[b], 1);
        mbar_init(&bars->p_full[b], 4);
    }
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

// As mma3, with a_lo a K-major shared-memory operand (128-row blocks `a_blk` bytes apart).
template <int N, int KS>
__device__ __forceinline__ void mma3_slo(uint32_t d, uint32_t a_hi, uint64_t a_lo, uint32_t a_blk, uint64_t b_hi,
                                         uint64_t b_lo, uint32_t blk)
{
    constexpr uint32_t idesc = idesc_tf32(BT, N);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const uint32_t off = (ks / 4) * blk + (ks % 4) * 32;
        mma_ts_tf32(d, a_hi + 8 * ks, sdesc_advance(b_hi, off), idesc, ks > 0 ? 1u : 0u);
        mma_ts_tf32(d, a_hi + 8 * ks, sdesc_advance(b_lo, off), idesc, 1u);
        mma_ss_tf32(d, sdesc_advance(a_lo, (ks / 4) * a_blk + (ks % 4) * 32), sdesc_advance(b_hi, off), idesc, 1u);
    }
}

// A streamed [BS rows x HD] fp32 tile goes from global memory (rows past S read as zero) into
// registers (load_tile, issued a tile ahead so the loads overlap the stores of the previous
// tile), then into a K-major hi / lo pair (`khi`, `klo`: HD / 32 blocks of BS rows x 128 B)
// and, when T, also its transpose (`thi`, `tlo`: HD rows x 128 B, the BS rows contiguous).
// 128 threads (warp w of the group, lane).  A warp takes 16 consecutive rows x 2 adjacent
// 16-byte columns: each row's 32 bytes are one sector of the global read, and with the
// 128-byte swizzle both the 16-byte K-major stores and the 4-byte transposed stores of a
// warp fall in distinct banks.
template <int HD>
struct TileRegs {
    static constexpr int N = BS * (HD / 4) / 128;   // 16-byte pieces per thread
    float4 x[N];
};

// Position of piece `it` of (warp w, lane): row r of the tile, 16-byte column c4.
template <int HD>
__device__ __forceinline__ void tile_pos(int it, int w, int lane, int &r, int &c4)
{
    constexpr int F4 = HD / 4;
    const int combo = it * 4 + w;                 // (16-row block, column pair)
    r = (combo / (F4 / 2)) * 16 + (lane & 15);
    c4 = (combo % (F4 / 2)) * 2 + (lane >> 4);
}

template <int HD>
__device__ __forceinline__ void load_tile(const float *src, int row0, int S, int w, int lane, TileRegs<HD> &t)
{
#pragma unroll
    for (int it = 0; it < TileRegs<HD>::N; ++it) {
        int r, c4;
        tile_pos<HD>(it, w, lane, r, c4);
        const bool valid = row0 + r < S;
        t.x[it] = ldg4_or_zero(src + (size_t)(valid ? row0 + r : 0) * HD + 4 * c4, valid);
    }
}

template <int HD, bool T>
__device__ __forceinline__ void store_tile(const TileRegs<HD> &t, int w, int lane, uint8_t *khi, uint8_t *klo,
                                           uint8_t *thi, uint8_t *tlo)
{
    constexpr uint32_t BLK = BS * 128;
#pragma unroll
    for (int it = 0; it < TileRegs<HD>::N; ++it) {
        int r, c4;
        tile_pos<HD>(it, w, lane, r, c4);
        float4 hi, lo;
        split4(t.x[it], hi, lo);
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
    static constexpr int NSK = HD == 64 ? 2 : 3;   // streamed-tile ring depth
    static constexpr int MAT = BS * HD * 4;        // one streamed operand tile
    static constexpr int OWN = BT * HD * 4;        // K_lo or V_lo of the CTA's 128 keys
    static constexpr int OWN_BLK = BT * 128;       // one 32-column block of those
    // K_lo, V_lo (K-major, the A operands of the lo products of S^T / dP^T), then the ring
    static constexpr int OFF_KLO = 0, OFF_VLO = OWN, OFF_RING = 2 * OWN;
    // stage: Q, dO (K-major, B of S^T / dP^T) and Q^T, dO^T (B of dK / dV), each as hi, lo
    static constexpr int OFF_QHI = 0, OFF_QLO = MAT, OFF_OHI = 2 * MAT, OFF_OLO = 3 * MAT;
    static constexpr int OFF_QTHI = 4 * MAT, OFF_QTLO = 5 * MAT, OFF_OTHI = 6 * MAT, OFF_OTLO = 7 * MAT;
    static constexpr int STAGE = 8 * MAT;
    static constexpr int OFF_SCR = OFF_RING + NSK * STAGE;   // per compute warp: 32 Lg + 32 D
    static constexpr int OFF_BAR = OFF_SCR + 4 * 64 * 4;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    // TMEM: K_hi, V_hi (A operands), two buffers of {S^T / P^T_hi, P^T_lo, dP^T / dS^T_hi, dS^T_lo}, dV, dK
    static constexpr uint32_t KHI = 0, VHI = HD, BUF0 = 2 * HD, DV = 2 * HD + 8 * BS, DK = DV + HD;
    static __device__ __forceinline__ uint32_t st(int b) { return BUF0 + 4 * BS * b; }
    static __device__ __forceinline__ uint32_t plo(int b) { return st(b) + BS; }
    static __device__ __forceinline__ uint32_t dpt(int b) { return st(b) + 2 * BS; }
    static __device__ __forceinline__ uint32_t dslo(int b) { return st(b) + 3 * BS; }
    static_assert(DK + HD <= 512, "TMEM columns");
    static_assert(NSK <= NS, "ring depth");
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
    constexpr int NSK = C::NSK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    uint8_t *ring = smem + C::OFF_RING;
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
            // thread = key: hi parts into TMEM, lo parts into the K-major shared tiles
            const int key = k0 + tid;
            const bool valid = key < S;
            const size_t roff = hoff + (size_t)min(key, S - 1) * HD;
            const uint32_t t = tmem + ((uint32_t)(w * 32) << 16);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float *src = (m == 0 ? K : V) + roff;
                uint8_t *lo_tile = smem + (m == 0 ? C::OFF_KLO : C::OFF_VLO);
#pragma unroll
                for (int c = 0; c < HD; c += 32) {
                    uint32_t hi[32];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float4 h4, l4;
                        split4(ldg4_or_zero(src + c + 4 * e, valid), h4, l4);
                        hi[4 * e] = __float_as_uint(h4.x);
                        hi[4 * e + 1] = __float_as_uint(h4.y);
                        hi[4 * e + 2] = __float_as_uint(h4.z);
                        hi[4 * e + 3] = __float_as_uint(h4.w);
                        const int c4 = c / 4 + e;
                        *reinterpret_cast<float4 *>(lo_tile + (c4 / 8) * C::OWN_BLK + sw128(tid, c4 % 8)) = l4;
                    }
                    tmem_st32(t + (m == 0 ? C::KHI : C::VHI) + c, hi);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->own_ready);
        }
        TileRegs<HD> xq, xo;
        load_tile<HD>(Q + hoff, k0, S, w, lane, xq);
        load_tile<HD>(dO + hoff, k0, S, w, lane, xo);
        for (int i = 0; i < nq; ++i) {
            const int st = i % NSK;
            if (i >= NSK && !warp_wait(&bars->empty[st], ((i / NSK) + 1) & 1, bars, status)) break;
            uint8_t *g = ring + st * C::STAGE;
            TileRegs<HD> nq_, no_;
            if (i + 1 < nq) {
                load_tile<HD>(Q + hoff, k0 + (i + 1) * BS, S, w, lane, nq_);
                load_tile<HD>(dO + hoff, k0 + (i + 1) * BS, S, w, lane, no_);
            }
            store_tile<HD, true>(xq, w, lane, g + C::OFF_QHI, g + C::OFF_QLO, g + C::OFF_QTHI, g + C::OFF_QTLO);
            store_tile<HD, true>(xo, w, lane, g + C::OFF_OHI, g + C::OFF_OLO, g + C::OFF_OTHI, g + C::OFF_OTLO);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[st]);
            xq = nq_;
            xo = no_;
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint32_t base = smem_u32(ring);
        auto desc = [&](int st, int off) { return sdesc_sw128(base + st * C::STAGE + off, 16, 1024); };
        const uint64_t d_klo = sdesc_sw128(smem_u32(smem + C::OFF_KLO), 16, 1024);
        const uint64_t d_vlo = sdesc_sw128(smem_u32(smem + C::OFF_VLO), 16, 1024);
        constexpr uint32_t BLK = BS * 128;
        // S^T = K Q^T and dP^T = V dO^T of tile i (stage st) into buffer b
        auto issue_scores = [&](int st, int b) {
            mma3_slo<BS, HD / 8>(tmem + C::st(b), tmem + C::KHI, d_klo, C::OWN_BLK, desc(st, C::OFF_QHI),
                                 desc(st, C::OFF_QLO), BLK);
            mma3_slo<BS, HD / 8>(tmem + C::dpt(b), tmem + C::VHI, d_vlo, C::OWN_BLK, desc(st, C::OFF_OHI),
                                 desc(st, C::OFF_OLO), BLK);
            tc_commit(&bars->s_full[b]);
        };
        bool ok = warp_wait(&bars->own_ready, 0, bars, status) && warp_wait(&bars->full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) issue_scores(0, 0);
            __syncwarp();
        }
        for (int i = 0; ok && i < nq; ++i) {
            if (i + 1 < nq) {
                // buffer (i+1)&1 last held tile i-1's P^T / dS^T, read by the dV / dK MMAs issued
                // before: the tensor pipe runs in order, so the overwrite follows that read
                const int sn = (i + 1) % NSK;
                if (!(ok = warp_wait(&bars->full[sn], ((i + 1) / NSK) & 1, bars, status))) break;
                tc_fence_after_sync();
                if (leader) issue_scores(sn, (i + 1) & 1);
                __syncwarp();
            }
            const int b = i & 1;
            if (!(ok = warp_wait(&bars->p_full[b], (i >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            const int st = i % NSK;
            if (leader) {
                // dV += P^T dO, dK += dS^T Q: K = the 32 query rows (one 128-byte block)
                mma3<HD, BS / 8>(tmem + C::DV, tmem + C::st(b), tmem + C::plo(b), desc(st, C::OFF_OTHI),
                                 desc(st, C::OFF_OTLO), 0, i > 0);
                mma3<HD, BS / 8>(tmem + C::DK, tmem + C::dpt(b), tmem + C::dslo(b), desc(st, C::OFF_QTHI),
                                 desc(st, C::OFF_QTLO), 0, i > 0);
                tc_commit(&bars->empty[st]);
                if (i == nq - 1) tc_commit(&bars->acc_done);
            }
            __syncwarp();
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
            const int q0 = k0 + i * BS, b = i & 1;
            __syncwarp();
            scr[lane] = lg_h[q0 + lane];          // rows past S: Lg = -inf, so p = 0
            scr[32 + lane] = d_h[q0 + lane];
            __syncwarp();
            if (!(ok = warp_wait(&bars->s_full[b], (i >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            uint32_t s[32], dp[32];
            tmem_ld32(t + C::st(b), s);
            tmem_ld32(t + C::dpt(b), dp);
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
            tmem_st32(t + C::st(b), p_hi);
            tmem_st32(t + C::plo(b), p_lo);
            tmem_st32(t + C::dpt(b), s);
            tmem_st32(t + C::dslo(b), dp);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[b]);
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
    // TMEM: Q, dO (hi, lo: A operands), two buffers of {S, dP / dS_hi, dS_lo}, dQ
    static constexpr uint32_t QHI = 0, QLO = HD, OHI = 2 * HD, OLO = 3 * HD, DQ = 4 * HD + 6 * BS;
    static __device__ __forceinline__ uint32_t sc(int b) { return 4 * HD + 3 * BS * b; }
    static __device__ __forceinline__ uint32_t dp(int b) { return sc(b) + BS; }
    static __device__ __forceinline__ uint32_t dslo(int b) { return sc(b) + 2 * BS; }
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
        TileRegs<HD> xk, xv;
        load_tile<HD>(K + hoff, 0, S, w, lane, xk);
        load_tile<HD>(V + hoff, 0, S, w, lane, xv);
        for (int j = 0; j < nk; ++j) {
            const int st = j % NS;
            if (j >= NS && !warp_wait(&bars->empty[st], ((j / NS) + 1) & 1, bars, status)) break;
            uint8_t *g = smem + st * C::STAGE;
            TileRegs<HD> nk_, nv_;
            if (j + 1 < nk) {
                load_tile<HD>(K + hoff, (j + 1) * BS, S, w, lane, nk_);
                load_tile<HD>(V + hoff, (j + 1) * BS, S, w, lane, nv_);
            }
            store_tile<HD, true>(xk, w, lane, g + C::OFF_KHI, g + C::OFF_KLO, g + C::OFF_KTHI, g + C::OFF_KTLO);
            store_tile<HD, false>(xv, w, lane, g + C::OFF_VHI, g + C::OFF_VLO, nullptr, nullptr);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[st]);
            xk = nk_;
            xv = nv_;
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint32_t base = smem_u32(smem);
        auto desc = [&](int st, int off) { return sdesc_sw128(base + st * C::STAGE + off, 16, 1024); };
        constexpr uint32_t BLK = BS * 128;
        // S = Q K^T and dP = dO V^T of the tile in stage st into buffer b
        auto issue_scores = [&](int st, int b) {
            mma3<BS, HD / 8>(tmem + C::sc(b), tmem + C::QHI, tmem + C::QLO, desc(st, C::OFF_KHI), desc(st, C::OFF_KLO),
                             BLK, false);
            mma3<BS, HD / 8>(tmem + C::dp(b), tmem + C::OHI, tmem + C::OLO, desc(st, C::OFF_VHI), desc(st, C::OFF_VLO),
                             BLK, false);
            tc_commit(&bars->s_full[b]);
        };
        bool ok = warp_wait(&bars->own_ready, 0, bars, status) && warp_wait(&bars->full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) issue_scores(0, 0);
            __syncwarp();
        }
        for (int j = 0; ok && j < nk; ++j) {
            if (j + 1 < nk) {
                // buffer (j+1)&1 last held tile j-1's dS, read by the dQ MMAs issued before (in order)
                const int sn = (j + 1) % NS;
                if (!(ok = warp_wait(&bars->full[sn], ((j + 1) / NS) & 1, bars, status))) break;
                tc_fence_after_sync();
                if (leader) issue_scores(sn, (j + 1) & 1);
                __syncwarp();
            }
            const int b = j & 1;
            if (!(ok = warp_wait(&bars->p_full[b], (j >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            const int st = j % NS;
            if (leader) {
                // dQ += dS K: A = dS_hi (over dP) / dS_lo, B = K^T (K = the 32 keys)
                mma3<HD, BS / 8>(tmem + C::DQ, tmem + C::dp(b), tmem + C::dslo(b), desc(st, C::OFF_KTHI),
                                 desc(st, C::OFF_KTLO), 0, j > 0);
                tc_commit(&bars->empty[st]);
                if (j == nk - 1) tc_commit(&bars->acc_done);
            }
            __syncwarp();
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
            const int b = j & 1;
            if (!(ok = warp_wait(&bars->s_full[b], (j >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            uint32_t s[32], dp[32];
            tmem_ld32(t + C::sc(b), s);
            tmem_ld32(t + C::dp(b), dp);
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
            tmem_st32(t + C::dp(b), s);
            tmem_st32(t + C::dslo(b), dp);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[b]);
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
