// 3xTF32 operand split and shared-memory tile layout of the fp32 tensor-core kernels
// (tf_fwd.cu, tf_bwd.cu).
//
// An fp32 value x is carried as hi + lo, both rounded to nearest tf32 in software
// (tf32_rna), so the tensor core reads them unchanged whatever its own handling of fp32
// inputs: hi = tf32(x), lo = tf32(x - hi) (x - hi is exact in fp32), |x - hi - lo| <=
// 2^-22 |x|.  A product a.b is formed as a_hi.b_hi + a_hi.b_lo + a_lo.b_hi by three
// kind::tf32 MMAs; the dropped a_lo.b_lo is below 2^-22 |a.b| as well, so each product
// carries about 2^-21 relative error against fp32's 2^-24.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace xfa {

// x rounded to the nearest tf32 value, ties away from zero (the rounding of cvt.rna.tf32.f32),
// done on the encoding: adding half a tf32 ulp (bit 12) to the magnitude bits and clearing the
// 13 bits below the tf32 mantissa rounds the magnitude half-up, a carry out of the mantissa
// steps the exponent, and infinities stay infinite.  Two integer operations instead of a
// conversion instruction.
__device__ __forceinline__ float tf32_rna(float x)
{
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo)
{
    const float h = tf32_rna(x);
    hi = __float_as_uint(h);
    lo = __float_as_uint(tf32_rna(x - h));
}

__device__ __forceinline__ void split4(const float4 &x, float4 &hi, float4 &lo)
{
    hi = make_float4(tf32_rna(x.x), tf32_rna(x.y), tf32_rna(x.z), tf32_rna(x.w));
    lo = make_float4(tf32_rna(x.x - hi.x), tf32_rna(x.y - hi.y), tf32_rna(x.z - hi.z), tf32_rna(x.w - hi.w));
}

// kind::tf32: D[tmem] (+)= A[tmem] * B[smem]  (A: M lanes x K fp32 elements, one per column;
// B: K-major, 128-byte rows of 32 elements).
__device__ __forceinline__ void mma_ts_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// kind::tf32: D[tmem] (+)= A[smem] * B[smem]^T  (both K-major, 128-byte rows of 32 elements).
__device__ __forceinline__ void mma_ss_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::tf32 with K-major tf32 A/B and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N)
{
    return (1u << 4)                       // D format: f32
           | (2u << 7)                     // A format: tf32
           | (2u << 10)                    // B format: tf32
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile of 128-byte rows with
// the 128-byte swizzle (chunk index XOR row mod 8; tile base 1024-byte aligned).  A K-major
// tcgen05 operand of 32-bit elements holds 32 of them per row.
__device__ __forceinline__ uint32_t sw128(int row, int chunk)
{
    return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

// Byte offset of 32-bit element `col` (0..31) of row `row` in the same layout.
__device__ __forceinline__ uint32_t sw128_word(int row, int col) { return sw128(row, col >> 2) + ((col & 3) << 2); }

__device__ __forceinline__ float4 ldg4_or_zero(const float *p, bool valid)
{
    return valid ? __ldg(reinterpret_cast<const float4 *>(p)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// One row of 32-bit values (thread = TMEM lane) from global memory into TMEM as hi / lo
// columns: `n` values starting at `src` (16-byte aligned), zeros when !valid.
template <int N>
__device__ __forceinline__ void row_to_tmem_split(const float *src, bool valid, uint32_t t_hi, uint32_t t_lo)
{
#pragma unroll
    for (int c = 0; c < N; c += 32) {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 x = ldg4_or_zero(src + c + 4 * e, valid);
            split_tf32(x.x, hi[4 * e + 0], lo[4 * e + 0]);
            split_tf32(x.y, hi[4 * e + 1], lo[4 * e + 1]);
            split_tf32(x.z, hi[4 * e + 2], lo[4 * e + 2]);
            split_tf32(x.w, hi[4 * e + 3], lo[4 * e + 3]);
        }
        tmem_st32(t_hi + c, hi);
        tmem_st32(t_lo + c, lo);
    }
}

}  // namespace xfa
