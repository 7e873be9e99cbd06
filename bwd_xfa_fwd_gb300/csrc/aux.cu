// Bandwidth kernels around the attention kernels:
//   - the backward pre-pass D_i = sum_d dO_i[d] O_i[d]
//     ("xtrain docs/13-flash-attention.md", design decision ③), fused with
//     the conversion of L to -L*log2(e), the padding of both arrays to whole
//     query tiles (so the backward kernels can bulk-copy them per tile) and
//     the clearing of the fp32 dQ accumulator;
//   - the fp32 dQ accumulator -> output dtype conversion;
//   - dst += src, the tape's fan-out gradient accumulation
//     ("xtrain docs/03-autograd-engine.md", section "梯度累加（扇出求和）");
//   - the timeout self-test kernel.
// Each row is read with 16-byte vector loads by a group of lanes and reduced
// with warp shuffles; grids are a multiple of the SM count.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace xfa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float dot16(const float4 &a, const float4 &b, float acc, float)
{
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    return fmaf(a.w, b.w, acc);
}

__device__ __forceinline__ float dot16(const uint4 &a, const uint4 &b, float acc, int)
{
    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 u = __bfloat1622float2(x[i]);
        const float2 v = __bfloat1622float2(y[i]);
        acc = fmaf(u.x, v.x, acc);
        acc = fmaf(u.y, v.y, acc);
    }
    return acc;
}

// VecT: float4 (fp32 storage) or uint4 (8 x bf16).  One row = HD elements.
template <typename VecT, int HD, int ELT, bool PREP>
__global__ void __launch_bounds__(256) rowdot_kernel(const VecT *__restrict__ O, const VecT *__restrict__ dO,
                                                     const float *__restrict__ lse, float *__restrict__ D,
                                                     float *__restrict__ Lg, float *__restrict__ zero_acc, int S,
                                                     int S_pad, long total_rows, float lg_bias)
{
    constexpr int VEC = 16 / ELT;      // elements per 16-byte vector
    constexpr int LPR = HD / VEC;      // lanes per row
    constexpr int RPW = 32 / LPR;      // rows per warp step
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    for (long base = warp * RPW; base < total_rows; base += nwarps * RPW) {
        const long r = base + lane / LPR;
        const bool valid = r < total_rows;
        const long b = valid ? r / S_pad : 0;
        const int i = valid ? (int)(r % S_pad) : 0;
        const bool real = valid && i < S;
        float acc = 0.0f;
        if (real) {
            const long v = ((b * S + i) * HD) / VEC + sub;
            acc = dot16(__ldg(O + v), __ldg(dO + v), 0.0f, (typename std::conditional<ELT == 4, float, int>::type)0);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid && sub == 0) {
            D[r] = acc;
            if (PREP) Lg[r] = real ? -lse[b * S + i] * kLog2e + lg_bias : -CUDART_INF_F;
        }
        if (PREP && real && zero_acc) {
            // clear this row of the fp32 dQ accumulator: HD floats over the LPR lanes of the row
            float4 *z = reinterpret_cast<float4 *>(zero_acc + (b * S + i) * HD);
#pragma unroll
            for (int e = sub; e < HD / 4; e += LPR) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

template <int HD>
cudaError_t rowdot_launch(const void *O, const void *dO, const float *lse, float *D, float *Lg, float *zero_acc,
                          int bh, int S, int S_pad, int dtype, bool prep, float lg_bias, cudaStream_t st)
{
    const long rows = (long)bh * S_pad;
    const int sms = sm_count();
    const long blocks_needed = (rows + 63) / 64;
    const unsigned grid = (unsigned)std::max<long>(1, std::min<long>(blocks_needed, (long)sms * 8));
    if (dtype == XFA_BF16) {
        if (prep)
            rowdot_kernel<uint4, HD, 2, true><<<grid, 256, 0, st>>>((const uint4 *)O, (const uint4 *)dO, lse, D, Lg,
                                                                     zero_acc, S, S_pad, rows, lg_bias);
        else
            rowdot_kernel<uint4, HD, 2, false><<<grid, 256, 0, st>>>((const uint4 *)O, (const uint4 *)dO, lse, D,
                                                                      Lg, zero_acc, S, S_pad, rows, lg_bias);
    } else {
        if (prep)
            rowdot_kernel<float4, HD, 4, true><<<grid, 256, 0, st>>>((const float4 *)O, (const float4 *)dO, lse, D,
                                                                      Lg, zero_acc, S, S_pad, rows, lg_bias);
        else
            rowdot_kernel<float4, HD, 4, false><<<grid, 256, 0, st>>>((const float4 *)O, (const float4 *)dO, lse,
                                                                       D, Lg, zero_acc, S, S_pad, rows, lg_bias);
    }
    return cudaGetLastError();
}

cudaError_t rowdot_any(const void *O, const void *dO, const float *lse, float *D, float *Lg, float *zero_acc, int bh,
                       int S, int S_pad, int hd, int dtype, bool prep, float lg_bias, cudaStream_t st)
{
    switch (hd) {
    case 32: return rowdot_launch<32>(O, dO, lse, D, Lg, zero_acc, bh, S, S_pad, dtype, prep, lg_bias, st);
    case 64: return rowdot_launch<64>(O, dO, lse, D, Lg, zero_acc, bh, S, S_pad, dtype, prep, lg_bias, st);
    case 128: return rowdot_launch<128>(O, dO, lse, D, Lg, zero_acc, bh, S, S_pad, dtype, prep, lg_bias, st);
    default: return cudaErrorInvalidValue;
    }
}

// fp32 -> bf16, four independent float4 per thread and step (loads issued first).
__global__ void __launch_bounds__(256) convert_bf16_kernel(const float4 *__restrict__ src, uint2 *__restrict__ dst,
                                                           size_t n4)
{
    constexpr int U = 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n4; i0 += U * stride) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u * stride < n4) v[u] = __ldg(src + i0 + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u * stride < n4) {
                uint2 o;
                o.x = pack_bf16x2(v[u].x, v[u].y);
                o.y = pack_bf16x2(v[u].z, v[u].w);
                dst[i0 + u * stride] = o;
            }
    }
}

__global__ void __launch_bounds__(256) copy_f32_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst,
                                                       size_t n4)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __ldg(src + i);
}

__global__ void __launch_bounds__(256) accumulate_f32_kernel(float *__restrict__ dst, const float *__restrict__ src,
                                                             size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] += src[i];
}

__global__ void __launch_bounds__(256) accumulate_bf16_kernel(__nv_bfloat16 *__restrict__ dst,
                                                              const __nv_bfloat16 *__restrict__ src, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __float2bfloat16_rn(__bfloat162float(dst[i]) + __bfloat162float(src[i]));
}

__global__ void selftest_timeout_kernel(uint64_t limit_ns, int *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: the wait must run out and report it.
    const bool ok = mbar_wait(&bar, 0, nullptr, limit_ns);
    if (!ok && threadIdx.x == 0) record_status(status, XFA_ERR_TIMEOUT);
}

unsigned elementwise_grid(size_t n)
{
    const size_t blocks = (n + 255) / 256;
    return (unsigned)std::max<size_t>(1, std::min<size_t>(blocks, (size_t)sm_count() * 16));
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdParams &p, cudaStream_t st)
{
    return rowdot_any(p.out, p.dout, p.lse, p.D, p.Lg, p.dq_acc, p.bh, p.S, p.S_pad, p.hd, p.dtype, true, p.lg_bias, st);
}

cudaError_t launch_rowdot(const void *out, const void *dout, float *d, int bh, int S, int hd, int dtype,
                          cudaStream_t st)
{
    return rowdot_any(out, dout, nullptr, d, nullptr, nullptr, bh, S, S, hd, dtype, false, 0.0f, st);
}

cudaError_t launch_convert_dq(const float *acc, void *dq, size_t n, int dtype, cudaStream_t st)
{
    const size_t n4 = n / 4;   // n = bh * S * hd with hd a multiple of 32
    if (dtype == XFA_BF16)
        convert_bf16_kernel<<<elementwise_grid(n4), 256, 0, st>>>((const float4 *)acc, (uint2 *)dq, n4);
    else
        copy_f32_kernel<<<elementwise_grid(n4), 256, 0, st>>>((const float4 *)acc, (float4 *)dq, n4);
    return cudaGetLastError();
}

cudaError_t launch_accumulate(void *dst, const void *src, size_t n, int dtype, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    if (dtype == XFA_BF16)
        accumulate_bf16_kernel<<<elementwise_grid(n), 256, 0, st>>>((__nv_bfloat16 *)dst,
                                                                     (const __nv_bfloat16 *)src, n);
    else
        accumulate_f32_kernel<<<elementwise_grid(n), 256, 0, st>>>((float *)dst, (const float *)src, n);
    return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned timeout_us, int *status, cudaStream_t st)
{
    selftest_timeout_kernel<<<1, 32, 0, st>>>((uint64_t)timeout_us * 1000ull, status);
    return cudaGetLastError();
}

}  // namespace xfa
