// SIMT (fp32 FFMA) flash-attention forward and backward.
//
// The fp32 workloads run here: tf32 tensor-core rounding (10-bit mantissa)
// cannot meet a 1e-4 relative tolerance, so these kernels keep every product
// in fp32.  They also accept bf16 storage and serve every hd in {32, 64, 128}.
//
// Forward ("xtrain docs/13-flash-attention.md", section "什么是 flash-attention"):
// a CTA owns a 64-row query tile of one head and scans the 64-key tiles at or
// below the diagonal with the online-softmax recurrence (running max m,
// running sum l, accumulator rescaled by exp(m_old - m_new)).  Unlike the
// page's one-block-per-row kernel, the K/V tile in shared memory is reused by
// 64 query rows.
//
// Backward (same section, and design decision ③): a CTA owns a 64-key tile,
// keeps its dK/dV rows in registers and walks the query tiles at or below the
// diagonal, recomputing p = exp(s - L) and ds = p (dp - D) scale; dQ rows are
// accumulated across key tiles with fp32 atomics.  This is the key-block-owned
// layout that the page lists as its follow-up for the dK/dV atomics.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "dropout.cuh"
#include "kernels.h"

namespace xfa {
namespace {

constexpr int kTile = 64;       // query rows and key rows per tile
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// rows [row0, row0 + kTile) of one head's [S][HD] matrix -> fp32 smem with row pitch `pitch`;
// rows at or beyond S read as zero.
template <typename T, int HD>
__device__ __forceinline__ void load_tile(float *dst, int pitch, const T *src, int row0, int S)
{
    for (int e = threadIdx.x; e < kTile * HD; e += kThreads) {
        const int r = e / HD, c = e % HD;
        const int row = row0 + r;
        dst[r * pitch + c] = row < S ? to_f32(src[(size_t)row * HD + c]) : 0.0f;
    }
}

template <typename T, int HD, bool DROP>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                           const T *__restrict__ V, T *__restrict__ O,
                                                           float *__restrict__ lse, int S, float scale_log2,
                                                           const DropParams drop)
{
    extern __shared__ float smem[];
    constexpr int KP = HD + 1;        // padded pitch for K (column walks)
    float *Qs = smem;                 // [64][HD]
    float *Ks = Qs + kTile * HD;      // [64][HD+1]
    float *Vs = Ks + kTile * KP;      // [64][HD]
    float *Ps = Vs + kTile * HD;      // [64][65]
    float *m_s = Ps + kTile * (kTile + 1);
    float *l_s = m_s + kTile;
    float *a_s = l_s + kTile;

    const int ntiles = (S + kTile - 1) / kTile;
    const int qt = ntiles - 1 - (int)(blockIdx.x % ntiles);   // heavy (long) rows first
    const size_t head = blockIdx.x / ntiles;
    const int q0 = qt * kTile;
    const T *Qh = Q + head * (size_t)S * HD;
    const T *Kh = K + head * (size_t)S * HD;
    const T *Vh = V + head * (size_t)S * HD;
    const int tid = threadIdx.x;

    load_tile<T, HD>(Qs, HD, Qh, q0, S);
    if (tid < kTile) {
        m_s[tid] = -CUDART_INF_F;
        l_s[tid] = 0.0f;
    }

    constexpr int CPT = HD / 4;       // output columns per thread
    float acc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[c] = 0.0f;
    const int orow = tid / 4, ocol = tid % 4;

    const int sr0 = (tid / 16) * 4, sc = tid % 16;   // score micro-tile: 4 rows x 4 strided cols

    for (int kt = 0; kt <= qt; ++kt) {
        const int k0 = kt * kTile;
        __syncthreads();
        load_tile<T, HD>(Ks, KP, Kh, k0, S);
        load_tile<T, HD>(Vs, HD, Vh, k0, S);
        __syncthreads();

        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.0f;
#pragma unroll 4
        for (int d = 0; d < HD; ++d) {
            float qv[4], kv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] = Qs[(sr0 + i) * HD + d];
#pragma unroll
            for (int j = 0; j < 4; ++j) kv[j] = Ks[(sc + 16 * j) * KP + d];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = sr0 + i, c = sc + 16 * j;
                const bool masked = (k0 + c) > (q0 + r);
                Ps[r * (kTile + 1) + c] = masked ? -CUDART_INF_F : s[i][j] * scale_log2;
            }
        __syncthreads();

        {   // online softmax statistics: 4 threads per row, 16 columns each
            const int r = tid / 4, part = tid % 4;
            float *prow = Ps + r * (kTile + 1) + part * 16;
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < 16; ++c) mx = fmaxf(mx, prow[c]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_old = m_s[r];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.0f;
            // dropout: the P.V product takes p o C (C_ij = keep / (1 - p)); the row sum keeps every p
            const uint64_t drop_g =
                DROP ? (((uint64_t)head * S + (uint64_t)(q0 + r)) * (uint64_t)S + (uint64_t)(k0 + part * 16)) *
                           kDropGolden
                     : 0ull;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p = exp2f(prow[c] - m_new);
                sum += p;
                if (DROP)
                    prow[c] = drop_keep(drop.seed, drop_g + (uint64_t)c * kDropGolden, drop.keep_thr) ? p * drop.inv_keep
                                                                                                     : 0.0f;
                else
                    prow[c] = p;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            __syncwarp();
            if (part == 0) {
                const float alpha = exp2f(m_old - m_new);
                a_s[r] = alpha;
                l_s[r] = l_s[r] * alpha + sum;
                m_s[r] = m_new;
            }
        }
        __syncthreads();

        const float alpha = a_s[orow];
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] *= alpha;
        const float *prow = Ps + orow * (kTile + 1);
#pragma unroll 4
        for (int j = 0; j < kTile; ++j) {
            const float p = prow[j];
            const float *vrow = Vs + j * HD + ocol;
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[c] = fmaf(p, vrow[4 * c], acc[c]);
        }
    }
    __syncthreads();

    const int row = q0 + orow;
    if (row < S) {
        const float inv_l = 1.0f / l_s[orow];
        T *orow_ptr = O + head * (size_t)S * HD + (size_t)row * HD + ocol;
#pragma unroll
        for (int c = 0; c < CPT; ++c) orow_ptr[4 * c] = from_f32<T>(acc[c] * inv_l);
        if (ocol == 0) lse[head * (size_t)S + row] = (m_s[orow] + log2f(l_s[orow])) * kLn2;
    }
}

template <typename T, int HD, bool DROP>
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                           const T *__restrict__ V, const T *__restrict__ dO,
                                                           const float *__restrict__ Lg, const float *__restrict__ Dv,
                                                           float *__restrict__ dQacc, T *__restrict__ dK,
                                                           T *__restrict__ dV, int S, int S_pad, float scale,
                                                           float scale_log2, const DropParams drop)
{
    extern __shared__ float smem[];
    constexpr int P = HD + 1;
    float *Ks = smem;                    // [64][HD+1]
    float *Vs = Ks + kTile * P;
    float *Qs = Vs + kTile * P;
    float *dOs = Qs + kTile * P;
    float *Ps = dOs + kTile * P;         // [64 q][65]
    float *dSs = Ps + kTile * (kTile + 1);
    float *Ls = dSs + kTile * (kTile + 1);
    float *Ds = Ls + kTile;

    const int ntiles = (S + kTile - 1) / kTile;
    const int kt = (int)(blockIdx.x % ntiles);       // low key tiles have the most query tiles: first
    const size_t head = blockIdx.x / ntiles;
    const int k0 = kt * kTile;
    const size_t hoff = head * (size_t)S * HD;
    const int tid = threadIdx.x;

    load_tile<T, HD>(Ks, P, K + hoff, k0, S);
    load_tile<T, HD>(Vs, P, V + hoff, k0, S);

    constexpr int CPT = HD / 4;
    float dk[CPT], dv[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) dk[c] = dv[c] = 0.0f;
    const int arow = tid / 4, acol = tid % 4;
    const int sr0 = (tid / 16) * 4, sc = tid % 16;   // (query rows, key cols) micro-tile

    for (int qt = kt; qt < ntiles; ++qt) {
        const int q0 = qt * kTile;
        __syncthreads();
        load_tile<T, HD>(Qs, P, Q + hoff, q0, S);
        load_tile<T, HD>(dOs, P, dO + hoff, q0, S);
        if (tid < kTile) {
            Ls[tid] = Lg[head * (size_t)S_pad + q0 + tid];
            Ds[tid] = Dv[head * (size_t)S_pad + q0 + tid];
        }
        __syncthreads();

        float s[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = dp[i][j] = 0.0f;
#pragma unroll 2
        for (int d = 0; d < HD; ++d) {
            float qv[4], ov[4], kv[4], vv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qv[i] = Qs[(sr0 + i) * P + d];
                ov[i] = dOs[(sr0 + i) * P + d];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kv[j] = Ks[(sc + 16 * j) * P + d];
                vv[j] = Vs[(sc + 16 * j) * P + d];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
                    dp[i][j] = fmaf(ov[i], vv[j], dp[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = sr0 + i, c = sc + 16 * j;
                const bool masked = (k0 + c) > (q0 + r);
                const float p = masked ? 0.0f : exp2f(fmaf(s[i][j], scale_log2, Ls[r]));
                if (DROP) {   // dV takes P o C; dS is formed from C o dP (the dropout node's backward)
                    const uint64_t g =
                        (((uint64_t)head * S + (uint64_t)(q0 + r)) * (uint64_t)S + (uint64_t)(k0 + c)) * kDropGolden;
                    const bool keep = drop_keep(drop.seed, g, drop.keep_thr);
                    Ps[r * (kTile + 1) + c] = keep ? p * drop.inv_keep : 0.0f;
                    dSs[r * (kTile + 1) + c] = p * ((keep ? dp[i][j] * drop.inv_keep : 0.0f) - Ds[r]) * scale;
                } else {
                    Ps[r * (kTile + 1) + c] = p;
                    dSs[r * (kTile + 1) + c] = p * (dp[i][j] - Ds[r]) * scale;
                }
            }
        __syncthreads();

        // dV_j += sum_i P_ij dO_i ; dK_j += sum_i dS_ij Q_i   (thread owns key row arow)
#pragma unroll 2
        for (int i = 0; i < kTile; ++i) {
            const float p = Ps[i * (kTile + 1) + arow];
            const float ds = dSs[i * (kTile + 1) + arow];
            const float *orow = dOs + i * P + acol;
            const float *qrow = Qs + i * P + acol;
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                dv[c] = fmaf(p, orow[4 * c], dv[c]);
                dk[c] = fmaf(ds, qrow[4 * c], dk[c]);
            }
        }
        // dQ_i += sum_j dS_ij K_j   (thread owns query row arow of this tile)
        const int qrow = q0 + arow;
        if (qrow < S) {
            float dq[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) dq[c] = 0.0f;
            const float *dsrow = dSs + arow * (kTile + 1);
#pragma unroll 2
            for (int j = 0; j < kTile; ++j) {
                const float ds = dsrow[j];
                const float *krow = Ks + j * P + acol;
#pragma unroll
                for (int c = 0; c < CPT; ++c) dq[c] = fmaf(ds, krow[4 * c], dq[c]);
            }
            float *dst = dQacc + hoff + (size_t)qrow * HD + acol;
#pragma unroll
            for (int c = 0; c < CPT; ++c) atomicAdd(dst + 4 * c, dq[c]);
        }
    }

    const int krow = k0 + arow;
    if (krow < S) {
        T *dkp = dK + hoff + (size_t)krow * HD + acol;
        T *dvp = dV + hoff + (size_t)krow * HD + acol;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            dkp[4 * c] = from_f32<T>(dk[c]);
            dvp[4 * c] = from_f32<T>(dv[c]);
        }
    }
}

template <typename T, int HD, bool DROP>
cudaError_t run_fwd(const FwdParams &p, cudaStream_t st)
{
    constexpr size_t smem = sizeof(float) * (kTile * HD * 2 + kTile * (HD + 1) + kTile * (kTile + 1) + 3 * kTile);
    auto kern = simt_fwd_kernel<T, HD, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int ntiles = (p.S + kTile - 1) / kTile;
    const unsigned grid = (unsigned)(ntiles * p.bh);
    kern<<<grid, kThreads, smem, st>>>((const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.out, p.lse, p.S,
                                       p.scale * kLog2e, p.drop);
    return cudaGetLastError();
}

template <typename T, int HD, bool DROP>
cudaError_t run_bwd(const BwdParams &p, cudaStream_t st)
{
    constexpr size_t smem = sizeof(float) * (4 * kTile * (HD + 1) + 2 * kTile * (kTile + 1) + 2 * kTile);
    auto kern = simt_bwd_kernel<T, HD, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int ntiles = (p.S + kTile - 1) / kTile;
    const unsigned grid = (unsigned)(ntiles * p.bh);
    kern<<<grid, kThreads, smem, st>>>((const T *)p.q, (const T *)p.k, (const T *)p.v, (const T *)p.dout, p.Lg,
                                       p.D, p.dq_acc, (T *)p.dk, (T *)p.dv, p.S, p.S_pad, p.scale,
                                       p.scale * kLog2e, p.drop);
    return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_dispatch(const FwdParams &p, cudaStream_t st)
{
    switch (p.hd) {
    case 32: return p.drop.on ? run_fwd<T, 32, true>(p, st) : run_fwd<T, 32, false>(p, st);
    case 64: return p.drop.on ? run_fwd<T, 64, true>(p, st) : run_fwd<T, 64, false>(p, st);
    case 128: return p.drop.on ? run_fwd<T, 128, true>(p, st) : run_fwd<T, 128, false>(p, st);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t bwd_dispatch(const BwdParams &p, cudaStream_t st)
{
    switch (p.hd) {
    case 32: return p.drop.on ? run_bwd<T, 32, true>(p, st) : run_bwd<T, 32, false>(p, st);
    case 64: return p.drop.on ? run_bwd<T, 64, true>(p, st) : run_bwd<T, 64, false>(p, st);
    case 128: return p.drop.on ? run_bwd<T, 128, true>(p, st) : run_bwd<T, 128, false>(p, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_simt_fwd(const FwdParams &p, cudaStream_t st)
{
    return p.dtype == XFA_BF16 ? fwd_dispatch<__nv_bfloat16>(p, st) : fwd_dispatch<float>(p, st);
}

cudaError_t launch_simt_bwd(const BwdParams &p, cudaStream_t st)
{
    return p.dtype == XFA_BF16 ? bwd_dispatch<__nv_bfloat16>(p, st) : bwd_dispatch<float>(p, st);
}

}  // namespace xfa
