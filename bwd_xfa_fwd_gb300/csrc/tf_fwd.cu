// Flash-attention forward for fp32 tensors on the sm_103a tensor cores (3xTF32).
//
// Method: "xtrain docs/13-flash-attention.md", section "什么是 flash-attention": for each
// query row, the online softmax over the key tiles at or below the diagonal (running max m,
// running sum l, accumulator rescaled by exp(m_old - m_new)), then out = acc / l and
// L = m + ln l.  This is the fp32 operator of the page's f32 entry point, computed on the
// tensor cores by the split of tf32x3.cuh instead of on FFMA.
//
// GB300 design:
//   * a CTA owns 128 query rows (MMA M) of one head and walks key tiles of 64 keys;
//   * warps 4-7 (split group) read Q once and every K and V tile straight from global memory
//     and split them: Q_hi, Q_lo into TMEM (the A operand of S; thread = row), K_hi, K_lo
//     into shared memory as K-major 128-byte-swizzled tiles, V transposed (V^T: hd rows of 64
//     keys, keys contiguous) as hi / lo -- every shared-memory operand is K-major;
//   * warp 8 issues the MMAs: S_j = Q K_j^T into one of two S buffers (S_{j+1} goes before
//     P_j V_j, so the softmax of tile j+1 overlaps the P.V of tile j) and O += P_j V_j with
//     P_hi, P_lo read from TMEM;
//   * warps 0-3 (softmax, thread = row) read S_j, update m and l, rescale O only when the
//     maximum grows by more than 2^8 (after waiting for the previous P.V), and write P_hi over
//     S_j and P_lo beside it.
// TMEM (512 columns): Q_hi [0,hd) Q_lo [hd,2hd) S_0 S_1 (64 each) P_lo,0 P_lo,1 (64 each) O (hd).
#include <math_constants.h>

#include "dropout.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tf32x3.cuh"

namespace xfa {
namespace {

constexpr int BM = 128;               // query rows per CTA (MMA M)
constexpr int BN = 64;                // keys per tile
constexpr int kThreads = 288;         // 9 warps
constexpr int kWarpSplit = 4, kWarpMma = 8;
constexpr int NS = 3;                 // depth of the split K / V^T ring
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int HD>
struct Cfg {
    static constexpr int KBLK = BN * 128;   // one 32-column block of a K tile (64 rows of 128 B)
    static constexpr int VBLK = HD * 128;   // one 32-key block of a V^T tile (hd rows of 128 B)
    static constexpr int MAT = BN * HD * 4; // one split operand tile
    static constexpr int OFF_KHI = 0, OFF_KLO = MAT, OFF_VHI = 2 * MAT, OFF_VLO = 3 * MAT;
    static constexpr int STAGE = 4 * MAT;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;   // barriers + alignment slack
    static constexpr uint32_t COL_QHI = 0, COL_QLO = HD, COL_O = 2 * HD + 256;
    static __device__ __forceinline__ uint32_t col_s(int b) { return 2 * HD + 64 * b; }
    static __device__ __forceinline__ uint32_t col_plo(int b) { return 2 * HD + 128 + 64 * b; }
    static_assert(COL_O + HD <= 512, "TMEM columns");
    static_assert(MAT == (HD / 32) * KBLK && MAT == (BN / 32) * VBLK, "tile sizes");
};

struct Bars {
    uint64_t q_full;                 // Q_hi, Q_lo in TMEM (one arrival per split warp)
    uint64_t kv_full[NS];            // split K / V^T stage written (one arrival per split warp)
    uint64_t kv_empty[NS];           // stage released (tensor-core commit after its P.V)
    uint64_t s_full[2];              // S buffer ready
    uint64_t p_full[2];              // P written (one arrival per softmax warp)
    uint64_t pv_done;                // one phase per P.V
    uint64_t o_full;                 // last P.V complete
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

// S = Q K^T (M=128, N=64, K=hd in steps of 8): A = Q_hi / Q_lo from TMEM, B = K_hi / K_lo.
template <int HD>
__device__ __forceinline__ void issue_s(uint32_t d, uint32_t q_hi, uint32_t q_lo, uint64_t k_hi, uint64_t k_lo)
{
    constexpr uint32_t idesc = idesc_tf32(BM, BN);
#pragma unroll
    for (int ks = 0; ks < HD / 8; ++ks) {
        const uint32_t off = (ks / 4) * Cfg<HD>::KBLK + (ks % 4) * 32;
        mma_ts_tf32(d, q_hi + 8 * ks, sdesc_advance(k_hi, off), idesc, ks > 0 ? 1u : 0u);
        mma_ts_tf32(d, q_hi + 8 * ks, sdesc_advance(k_lo, off), idesc, 1u);
        mma_ts_tf32(d, q_lo + 8 * ks, sdesc_advance(k_hi, off), idesc, 1u);
    }
}

// O += P V (M=128, N=hd, K=64 keys in steps of 8): A = P_hi / P_lo from TMEM, B = V^T_hi / V^T_lo.
template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t o, uint32_t p_hi, uint32_t p_lo, uint64_t v_hi, uint64_t v_lo,
                                         bool accumulate)
{
    constexpr uint32_t idesc = idesc_tf32(BM, HD);
#pragma unroll
    for (int ks = 0; ks < BN / 8; ++ks) {
        const uint32_t off = (ks / 4) * Cfg<HD>::VBLK + (ks % 4) * 32;
        mma_ts_tf32(o, p_hi + 8 * ks, sdesc_advance(v_hi, off), idesc, (accumulate || ks > 0) ? 1u : 0u);
        mma_ts_tf32(o, p_hi + 8 * ks, sdesc_advance(v_lo, off), idesc, 1u);
        mma_ts_tf32(o, p_lo + 8 * ks, sdesc_advance(v_hi, off), idesc, 1u);
    }
}

// DROP: dropout on the probabilities that enter P.V (the row sums l keep every p).
template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    tf_fwd_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                  float *__restrict__ O, float *__restrict__ lse, int bh, int S, float scale_log2, int *status,
                  const DropParams drop)
{
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int nqt = (S + BM - 1) / BM;
    const int qt = nqt - 1 - (int)blockIdx.x / bh;   // longest query tiles first
    const int head = (int)blockIdx.x % bh;
    const int q0 = qt * BM;
    const int n = (min(S, q0 + BM) + BN - 1) / BN;   // key tiles at or below the diagonal

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 4);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->kv_full[s], 4);
            mbar_init(&bars->kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->s_full[b], 1);
            mbar_init(&bars->p_full[b], 4);
        }
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->drain, 1);
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

    if (warp >= kWarpSplit && warp < kWarpMma) {
        const int w = warp - kWarpSplit;              // TMEM lane quarter of this warp
        const int tid = threadIdx.x - kWarpSplit * 32;
        {
            const int row = q0 + tid;
            const uint32_t lane_off = (uint32_t)(w * 32) << 16;
            row_to_tmem_split<HD>(Q + ((size_t)head * S + min(row, S - 1)) * HD, row < S,
                                  tmem + lane_off + C::COL_QHI, tmem + lane_off + C::COL_QLO);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->q_full);
        }
        constexpr int F4 = HD / 4;   // 16-byte pieces per row
        for (int j = 0; j < n; ++j) {
            const int st = j % NS;
            if (j >= NS && !warp_wait(&bars->kv_empty[st], ((j / NS) + 1) & 1, bars, status)) break;
            uint8_t *stage = smem + st * C::STAGE;
            const int key0 = j * BN;
            // K: consecutive threads along a key row; one 16-byte chunk each into K_hi / K_lo
#pragma unroll
            for (int it = 0; it < BN * F4 / 128; ++it) {
                const int idx = it * 128 + tid;
                const int key = idx / F4, c4 = idx % F4;
                const bool valid = key0 + key < S;
                const float4 x = ldg4_or_zero(K + ((size_t)head * S + (valid ? key0 + key : 0)) * HD + 4 * c4, valid);
                float4 hi, lo;
                split4(x, hi, lo);
                const uint32_t off = (c4 / 8) * C::KBLK + sw128(key, c4 % 8);
                *reinterpret_cast<float4 *>(stage + C::OFF_KHI + off) = hi;
                *reinterpret_cast<float4 *>(stage + C::OFF_KLO + off) = lo;
            }
            // V^T: lane = key within a 32-key block, so each store of a column d fills one
            // 128-byte row of V^T (no bank conflicts); the warp's items are (block, 4 columns)
#pragma unroll
            for (int it = 0; it < HD / 8; ++it) {
                const int item = w * (HD / 8) + it;
                const int kb = item / F4, d4 = item % F4;
                const int key = kb * 32 + lane;
                const bool valid = key0 + key < S;
                const float4 x = ldg4_or_zero(V + ((size_t)head * S + (valid ? key0 + key : 0)) * HD + 4 * d4, valid);
                float4 hi, lo;
                split4(x, hi, lo);
                const float hs[4] = {hi.x, hi.y, hi.z, hi.w}, ls[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t off = kb * C::VBLK + sw128_word(4 * d4 + e, lane);
                    *reinterpret_cast<float *>(stage + C::OFF_VHI + off) = hs[e];
                    *reinterpret_cast<float *>(stage + C::OFF_VLO + off) = ls[e];
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->kv_full[st]);
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint32_t base = smem_u32(smem);
        const uint64_t d_khi = sdesc_sw128(base + C::OFF_KHI, 16, 1024);
        const uint64_t d_klo = sdesc_sw128(base + C::OFF_KLO, 16, 1024);
        const uint64_t d_vhi = sdesc_sw128(base + C::OFF_VHI, 16, 1024);
        const uint64_t d_vlo = sdesc_sw128(base + C::OFF_VLO, 16, 1024);
        bool ok = warp_wait(&bars->q_full, 0, bars, status) && warp_wait(&bars->kv_full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) {
                issue_s<HD>(tmem + C::col_s(0), tmem + C::COL_QHI, tmem + C::COL_QLO, d_khi, d_klo);
                tc_commit(&bars->s_full[0]);
            }
            __syncwarp();
        }
        for (int j = 0; ok && j < n; ++j) {
            const int jn = j + 1;
            if (jn < n) {
                const int stn = jn % NS;
                if (!(ok = warp_wait(&bars->kv_full[stn], (jn / NS) & 1, bars, status))) break;
                tc_fence_after_sync();
                if (leader) {
                    // S buffer jn & 1 last held P_{j-1}, whose P.V was issued before: the tensor
                    // pipe runs in order, so this overwrite follows that read
                    issue_s<HD>(tmem + C::col_s(jn & 1), tmem + C::COL_QHI, tmem + C::COL_QLO,
                                sdesc_advance(d_khi, stn * C::STAGE), sdesc_advance(d_klo, stn * C::STAGE));
                    tc_commit(&bars->s_full[jn & 1]);
                }
                __syncwarp();
            }
            if (!(ok = warp_wait(&bars->p_full[j & 1], (j >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            if (leader) {
                const int st = j % NS;
                issue_pv<HD>(tmem + C::COL_O, tmem + C::col_s(j & 1), tmem + C::col_plo(j & 1),
                             sdesc_advance(d_vhi, st * C::STAGE), sdesc_advance(d_vlo, st * C::STAGE), j > 0);
                tc_commit(&bars->pv_done);
                tc_commit(&bars->kv_empty[st]);
                if (j == n - 1) tc_commit(&bars->o_full);
            }
            __syncwarp();
        }
        if (leader) {
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0, nullptr);
        }
        __syncwarp();
    } else {
        // softmax, thread = query row (TMEM lane)
        const int r = warp * 32 + lane, row = q0 + r;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float m = -CUDART_INF_F, l = 0.0f;
        bool ok = true;
        // dropout: element (row, key) has flat index (head*S + row)*S + key
        const uint64_t drop_row_g = DROP ? ((uint64_t)head * S + (uint64_t)row) * (uint64_t)S * kDropGolden : 0ull;
        for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            if (!(ok = warp_wait(&bars->s_full[b], (j >> 1) & 1, bars, status))) break;
            tc_fence_after_sync();
            uint32_t s[BN];
            tmem_ld32(tmem + lane_off + C::col_s(b), s);
            tmem_ld32(tmem + lane_off + C::col_s(b) + 32, s + 32);
            tmem_wait_ld();
            reg_fence32(s);
            reg_fence32(s + 32);
            const int kmax = row - j * BN;   // columns past this are keys after the row
            if (kmax < BN - 1) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c > kmax) s[c] = 0xff800000u;   // -inf
            }
            float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
            for (int c = 0; c < BN; c += 8)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    mx4[e] = fmax3(mx4[e], __uint_as_float(s[c + 2 * e]), __uint_as_float(s[c + 2 * e + 1]));
            const float mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            const float m_new = fmaxf(m, mx * scale_log2);   // scale > 0: max commutes with the scaling
            if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                const float alpha = ex2_approx(m - m_new);   // 0 on the first tile
                l *= alpha;
                if (j > 0) {
                    // O holds P_{j-1} V_{j-1} only once that P.V has completed (S_j was issued
                    // after P_{j-2} V_{j-2}, so at most this one phase is outstanding)
                    if (!(ok = warp_wait(&bars->pv_done, (j - 1) & 1, bars, status))) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < HD; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + C::COL_O + c, o);
                        tmem_wait_ld();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_off + C::COL_O + c, o);
                    }
                }
                m = m_new;
            }
            float l4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            uint64_t drop_g = DROP ? drop_row_g + (uint64_t)(j * BN) * kDropGolden : 0ull;
#pragma unroll
            for (int h = 0; h < BN / 32; ++h) {
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float p = ex2_approx(fmaf(__uint_as_float(s[32 * h + e]), scale_log2, -m));
                    l4[e & 3] += p;
                    if (DROP) {
                        p = drop_keep(drop.seed, drop_g, drop.keep_thr) ? p * drop.inv_keep : 0.0f;
                        drop_g += kDropGolden;
                    }
                    split_tf32(p, hi[e], lo[e]);
                }
                tmem_st32(tmem + lane_off + C::col_s(b) + 32 * h, hi);
                tmem_st32(tmem + lane_off + C::col_plo(b) + 32 * h, lo);
            }
            l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[b]);
        }
        if (ok && warp_wait(&bars->o_full, 0, bars, status)) {
            tc_fence_after_sync();
            const float inv_l = 1.0f / l;
            float *orow = O + ((size_t)head * S + min(row, S - 1)) * HD;
#pragma unroll 1
            for (int c = 0; c < HD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + C::COL_O + c, o);
                tmem_wait_ld();
                reg_fence32(o);
                if (row < S) {
                    float4 *dst = reinterpret_cast<float4 *>(orow + c);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                             __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
                }
            }
            if (row < S) lse[(size_t)head * S + row] = (m + __log2f(l)) * kLn2;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <int HD, bool DROP>
int run(const FwdParams &p, cudaStream_t st)
{
    static_assert(Cfg<HD>::SMEM <= 227 * 1024, "shared memory per CTA");
    auto kern = tf_fwd_kernel<HD, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<HD>::SMEM);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    const unsigned grid = (unsigned)(((p.S + BM - 1) / BM) * p.bh);
    kern<<<grid, kThreads, Cfg<HD>::SMEM, st>>>((const float *)p.q, (const float *)p.k, (const float *)p.v,
                                                 (float *)p.out, p.lse, p.bh, p.S, p.scale * 1.4426950408889634f,
                                                 p.status, p.drop);
    e = cudaGetLastError();
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

}  // namespace

int launch_tf_fwd(const FwdParams &p, cudaStream_t st)
{
    if (p.dtype != XFA_F32) return XFA_ERR_UNSUPPORTED;
    if (p.hd == 64) return p.drop.on ? run<64, true>(p, st) : run<64, false>(p, st);
    if (p.hd == 32) return p.drop.on ? run<32, true>(p, st) : run<32, false>(p, st);
    return XFA_ERR_UNSUPPORTED;
}

}  // namespace xfa
