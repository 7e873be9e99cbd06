// dQ of the flash-attention backward as its own query-tile-parallel pass on the
// sm_103a tensor cores: no atomics, so the backward is bit-reproducible.
//
// Method: "xtrain docs/13-flash-attention.md", section "什么是 flash-attention":
// dQ_i = sum_j ds_ij K_j with p_ij = exp(s_ij - L_i), dp_ij = dO_i . V_j and
// ds_ij = p_ij (dp_ij - D_i) scale.  The page's own kernel keeps dQ private to
// the query row's block; here a CTA owns 128 query rows of one head, keeps
// dQ in TMEM across every key tile at or below the diagonal, and writes it once.
//
// GB300 design:
//   * warp 4 loads Q_i and dO_i once and streams K_j, V_j through a TMA ring;
//   * warp 5 (one elected lane) issues, per key tile j:
//       S   = Q_i K_j^T    (M=128 rows, N=128 keys, K=hd)  -> TMEM, double buffered
//       dP  = dO_i V_j^T   (M=128, N=128, K=hd)            -> TMEM
//       dQ += dS K_j       (A = dS bf16 in the S columns, B = K_j MN-major)
//   * warps 0-3 (thread = query row; L and D of the row stay in registers)
//     turn S and dP into dS = 2^(s scale log2e - L log2e) (dP - D) scale and
//     write it back as bf16 into the S columns;
//   * the epilogue converts the dQ rows to the output dtype.
// TMEM map (512 columns): S x2 [0,256) dP [256,384) dQ [384,384+hd).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace xfa {
namespace {

constexpr int BM = 128;                 // query rows per CTA (MMA M)
constexpr int BN = 128;                 // keys per tile
constexpr int kThreads = 192;           // 4 compute warps, TMA warp, MMA warp
constexpr int kWarpTma = 4, kWarpMma = 5;
constexpr int kHeadBundle = 8;

template <int HD>
struct Cfg {
    static constexpr int SUB = HD / 64;
    static constexpr int SUB_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = 128 * HD * 2;
    static constexpr int NS = HD == 128 ? 2 : 3;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = TILE_BYTES;
    static constexpr int OFF_K = 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static constexpr uint32_t COL_S = 0, COL_DP = 256, COL_DQ = 384;
};

struct Bars {
    uint64_t qdo_full;
    uint64_t k_full[3], v_full[3], kv_empty[3];
    uint64_t dp_full, ds_full, done, drain;   // dp_full: S and dP of a key tile in TMEM
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
    bool ok = mbar_wait_spin(bar, parity, &b->abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) fail(b, status);
    return ok;
}

// C[M=128, N=128] = A[128 x hd] * B[128 x hd]^T, both K-major (hd contiguous, 128-byte swizzle).
template <int HD>
__device__ __forceinline__ void issue_rows_dot(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc)
{
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
        const uint32_t off = (ks / 4) * Cfg<HD>::SUB_BYTES + (ks % 4) * 32;
        mma_ss(d_tmem, sdesc_advance(a_desc, off), sdesc_advance(b_desc, off), idesc, ks > 0);
    }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    tc_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const float *__restrict__ Lg, const float *__restrict__ Dg, __nv_bfloat16 *__restrict__ dQ, int bh,
                 int S, int S_pad, float scale, float scale_log2, int *status, int bundle_heads)
{
    using C = Cfg<HD>;
    static_assert(sizeof(Bars) <= 256, "barrier block");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // heads in bundles of bundle_heads (see head_bundle), longest query tiles first within a bundle
    const int nqt = (S + BM - 1) / BM;
    const int bundle = (int)blockIdx.x / (nqt * bundle_heads);
    const int g = min(bundle_heads, bh - bundle * bundle_heads);
    const int idx = (int)blockIdx.x - bundle * nqt * bundle_heads;
    const int qt = nqt - 1 - idx / g;
    const int head = bundle * bundle_heads + idx % g;
    const int q0 = qt * BM;
    const int nkv = qt + 1;   // key tiles 0..qt (tile qt holds the diagonal)

    if (threadIdx.x == 0) {
        mbar_init(&bars->qdo_full, 1);
        for (int s = 0; s < 3; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->ds_full, 4);   // one arrival per compute warp
        mbar_init(&bars->done, 1);
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

    if (warp == kWarpTma) {
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_do);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(&bars->qdo_full, 2 * C::TILE_BYTES);
            for (int s = 0; s < C::SUB; ++s) {
                tma_load_3d(smem + C::OFF_Q + s * C::SUB_BYTES, &tm_q, &bars->qdo_full, s * 64, q0, head);
                tma_load_3d(smem + C::OFF_DO + s * C::SUB_BYTES, &tm_do, &bars->qdo_full, s * 64, q0, head);
            }
            int issued[3] = {0, 0, 0};
            for (int j = 0; j < nkv; ++j) {
                const int st = j % C::NS;
                if (j >= C::NS && !mbar_wait_spin(&bars->kv_empty[st], ((j / C::NS) + 1) & 1, &bars->abort)) {
                    fail(bars, status);
                    break;
                }
                mbar_arrive_expect_tx(&bars->k_full[st], C::TILE_BYTES);
                for (int s = 0; s < C::SUB; ++s)
                    tma_load_3d(smem + C::OFF_K + st * C::TILE_BYTES + s * C::SUB_BYTES, &tm_k, &bars->k_full[st],
                                s * 64, j * BN, head);
                mbar_arrive_expect_tx(&bars->v_full[st], C::TILE_BYTES);
                for (int s = 0; s < C::SUB; ++s)
                    tma_load_3d(smem + C::OFF_V + st * C::TILE_BYTES + s * C::SUB_BYTES, &tm_v, &bars->v_full[st],
                                s * 64, j * BN, head);
                issued[st] = j + 1;
            }
            // never leave the CTA with copies in flight
            mbar_wait_spin(&bars->qdo_full, 0, nullptr);
            for (int st = 0; st < C::NS; ++st) {
                if (issued[st] == 0) continue;
                const uint32_t ph = ((issued[st] - 1) / C::NS) & 1;
                mbar_wait_spin(&bars->k_full[st], ph, nullptr);
                mbar_wait_spin(&bars->v_full[st], ph, nullptr);
            }
        }
    } else if (warp == kWarpMma) {
        const bool leader = elect_one();
        const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
        const uint64_t do_desc = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
        const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
        const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
        const uint64_t k_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::SUB_BYTES, 1024);   // K_j as an MN-major B
        constexpr uint32_t idesc_dq = idesc_bf16(BM, HD, false, true);
        bool ok = warp_wait(&bars->qdo_full, 0, bars, status) && warp_wait(&bars->k_full[0], 0, bars, status) &&
                  warp_wait(&bars->v_full[0], 0, bars, status);
        if (ok) {
            tc_fence_after_sync();
            if (leader) {
                issue_rows_dot<HD>(tmem + C::COL_S, q_desc, k_desc);
                issue_rows_dot<HD>(tmem + C::COL_DP, do_desc, v_desc);
                tc_commit(&bars->dp_full);
            }
            __syncwarp();
        }
        for (int j = 0; ok && j < nkv; ++j) {
            const int st = j % C::NS, jn = j + 1, stn = jn % C::NS;
            const uint32_t phn = (jn / C::NS) & 1;
            if (jn < nkv) {   // next S into the other buffer; its dS was consumed by the previous dQ MMA
                if (!(ok = warp_wait(&bars->k_full[stn], phn, bars, status))) break;
                tc_fence_after_sync();
                if (leader) {
                    issue_rows_dot<HD>(tmem + C::COL_S + 128 * (jn & 1), q_desc, sdesc_advance(k_desc, stn * C::TILE_BYTES));
                }
                __syncwarp();
            }
            if (!(ok = warp_wait(&bars->ds_full, j & 1, bars, status))) break;
            if (jn < nkv && !(ok = warp_wait(&bars->v_full[stn], phn, bars, status))) break;
            tc_fence_after_sync();
            if (leader) {
                if (jn < nkv) {   // dP was read before dS was written: its columns are free
                    issue_rows_dot<HD>(tmem + C::COL_DP, do_desc, sdesc_advance(v_desc, stn * C::TILE_BYTES));
                    tc_commit(&bars->dp_full);
                }
                // dQ += dS K_j: dS (bf16 pairs) in the first 64 columns of its S buffer; 16 keys per step
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    mma_ts(tmem + C::COL_DQ, tmem + C::COL_S + 128 * (j & 1) + ks * 8,
                           sdesc_advance(k_mn, st * C::TILE_BYTES + ks * 2048), idesc_dq, (j > 0 || ks > 0) ? 1u : 0u);
                tc_commit(&bars->kv_empty[st]);
            }
            __syncwarp();
        }
        if (leader) {
            if (ok) tc_commit(&bars->done);
            tc_commit(&bars->drain);
            mbar_wait_spin(&bars->drain, 0, nullptr);
        }
        __syncwarp();
    } else {
        // compute warps: thread = query row r (TMEM lane)
        const int r = warp * 32 + lane;
        const int row = q0 + r;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float negl = Lg[(size_t)head * S_pad + row];   // -L * log2(e); -inf on padded rows
        const float dd = Dg[(size_t)head * S_pad + row];
        const uint64_t cs2 = f2_pack(scale_log2, scale_log2);
        const uint64_t nl2 = f2_pack(negl, negl);
        const uint64_t nd2 = f2_pack(-dd, -dd);
        const uint64_t sc2 = f2_pack(scale, scale);
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            // dP of this tile is issued after its S (the S of tile j goes out before tile j - 1's dS
            // is waited for, this tile's dP after it), so the dP commit also covers the S: one wait
            if (!(ok = warp_wait(&bars->dp_full, j & 1, bars, status))) break;
            tc_fence_after_sync();
            const uint32_t tS = tmem + lane_off + C::COL_S + 128 * (j & 1);
            const uint32_t tP = tmem + lane_off + C::COL_DP;
            const bool diag = j == qt;
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // 32 keys at a time
                uint32_t sr[32], dp[32];
                tmem_ld32(tS + 32 * k, sr);
                tmem_ld32(tP + 32 * k, dp);
                tmem_wait_ld();
                reg_fence32(sr);
                reg_fence32(dp);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c = 32 * k + 2 * e;   // key index within the tile
                    const float2 a = f2_unpack(ffma2(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                                                     cs2, nl2));
                    float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
                    if (diag) {
                        if (c > r) p0 = 0.0f;
                        if (c + 1 > r) p1 = 0.0f;
                    }
                    const uint64_t t = fadd2(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), nd2);
                    const float2 ds = f2_unpack(fmul2(fmul2(f2_pack(p0, p1), sc2), t));
                    pk[e] = pack_bf16x2(ds.x, ds.y);
                }
                // dS pairs overwrite S columns already read (chunk k writes [16k, 16k+16) <= read range)
                tmem_st16(tS + 16 * k, pk);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->ds_full);
        }
        if (ok && warp_wait(&bars->done, 0, bars, status)) {
            tc_fence_after_sync();
            __nv_bfloat16 *dst = dQ + ((size_t)head * S + row) * HD;
#pragma unroll 1
            for (int c = 0; c < HD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + C::COL_DQ + c, o);
                tmem_wait_ld();
                reg_fence32(o);
                if (row < S) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]), __uint_as_float(o[8 * v + 1]));
                        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3]));
                        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5]));
                        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7]));
                        reinterpret_cast<uint4 *>(dst + c)[v] = w;
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <int HD>
int run(const BwdParams &p, cudaStream_t st)
{
    alignas(64) CUtensorMap tq, tdo, tk, tv;
    int rc = encode_tmap_bf16_3d(&tq, p.q, HD, p.S, p.bh, BM);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tdo, p.dout, HD, p.S, p.bh, BM);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tk, p.k, HD, p.S, p.bh, BN);
    if (rc == XFA_OK) rc = encode_tmap_bf16_3d(&tv, p.v, HD, p.S, p.bh, BN);
    if (rc != XFA_OK) return rc;
    static_assert(Cfg<HD>::SMEM <= 227 * 1024, "shared memory per CTA");
    auto kern = tc_dq_kernel<HD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<HD>::SMEM);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    const int nqt = (p.S + BM - 1) / BM;
    kern<<<(unsigned)(nqt * p.bh), kThreads, Cfg<HD>::SMEM, st>>>(tq, tdo, tk, tv, p.Lg, p.D,
                                                                   (__nv_bfloat16 *)p.dq, p.bh, p.S, p.S_pad, p.scale,
                                                                   p.scale * 1.4426950408889634f, p.status,
                                                                   head_bundle(p.bh, p.S, HD, 2, kHeadBundle));
    e = cudaGetLastError();
    return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e;
}

}  // namespace

int launch_tc_dq(const BwdParams &p, cudaStream_t st)
{
    if (p.dtype != XFA_BF16) return XFA_ERR_UNSUPPORTED;
    if (p.hd == 128) return run<128>(p, st);
    if (p.hd == 64) return run<64>(p, st);
    return XFA_ERR_UNSUPPORTED;
}

}  // namespace xfa
