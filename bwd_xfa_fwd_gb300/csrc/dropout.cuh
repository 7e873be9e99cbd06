// Counter-based dropout draw of "xtrain docs/17-dropout.md", section "Key Design
// Decisions": element idx of a tensor is kept when u >= p, with
//   key = seed XOR (idx * 0x9E3779B97F4A7C15),  h = splitmix64(key),  u = (h >> 40) / 2^24,
// where splitmix64(x) is one step of the SplitMix64 generator (Steele, Lea and Flood,
// OOPSLA 2014) from state x: add the golden-ratio increment, then the two
// xor-shift-multiply rounds and a final xor-shift.  The final xor-shift (z ^ (z >> 31))
// does not change the top 24 bits, so the draw stops before it.  No state: the same
// (seed, idx) gives the same decision in the forward and in the backward.
#pragma once

#include <cstdint>

namespace xfa {

constexpr uint64_t kDropGolden = 0x9E3779B97F4A7C15ull;

// Top 24 bits of splitmix64(key).
__device__ __forceinline__ uint32_t drop_draw24(uint64_t key)
{
    uint64_t z = key + kDropGolden;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)(z >> 40);
}

// Keep decision of the element whose flat index times the golden ratio (mod 2^64) is
// idx_golden; kernels step idx_golden by a constant along a row instead of multiplying.
__device__ __forceinline__ bool drop_keep(uint64_t seed, uint64_t idx_golden, uint32_t keep_thr)
{
    return drop_draw24(seed ^ idx_golden) >= keep_thr;
}

}  // namespace xfa
