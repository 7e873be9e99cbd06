// Filling the cached keep bits of dropout on the attention probabilities.
//
// Method: "xtrain docs/17-dropout.md", sections "Goal" and "Key Design Decisions": the mask is
// generated once from (seed, element index) by the counter-based draw and the forward and the
// backward both apply that same mask.  Here the generation is a kernel of its own, so that it can
// run ahead of the attention (on another stream, or while other work runs) and both attention
// kernels only read its bits.
//
// Layout (keep_word in dropout.cuh): bit i of word ((b * nkt + kt) * nw + w) * 128 + c is the
// decision of probability (b, query row 32 w + i, key 128 kt + c).  Every word at or below the
// diagonal block of its key tile (4 kt <= w < nw) is written -- the words the forward kernel writes
// when it draws for itself, bit for bit, rows and keys past S included.
#include "dropout.cuh"
#include "kernels.h"

namespace xfa {
namespace {

// Block = (b, kt) x R chunks of 4 word rows: thread = key c, word row w = 4 chunk + y of each of
// its R chunks, 32 draws per word; chunks wholly above the diagonal block are skipped.  Large
// grids take R = 4 (fewer, longer blocks: 4 % faster at bh 32, S 8192), small ones R = 1 (enough
// blocks to fill the SMs: R = 4 was 10 % slower at bh 96, S 1024).
template <int kFillChunks>
__global__ void __launch_bounds__(512) keep_fill_kernel(uint32_t *__restrict__ keep, int S, int nkt, int nw,
                                                        uint64_t seed, uint32_t keep_thr)
{
    const int b = (int)blockIdx.x / nkt, kt = (int)blockIdx.x % nkt;
    const int chunk0 = kFillChunks * (int)blockIdx.y, c = threadIdx.x;
    if (chunk0 + kFillChunks <= kt) return;
    const uint64_t key = (uint64_t)(kt * 128 + c);
    const uint64_t step = (uint64_t)S * kDropGolden;   // the next row, same key
#pragma unroll 1
    for (int r = 0; r < kFillChunks; ++r) {
        const int chunk = chunk0 + r;
        if (chunk < kt || chunk >= nkt) continue;
        const int w = 4 * chunk + (int)threadIdx.y;
        uint64_t g = (((uint64_t)b * S + 32u * (uint64_t)w) * (uint64_t)S + key) * kDropGolden;
        uint32_t bits = 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            bits |= (uint32_t)drop_keep(seed, g, keep_thr) << i;
            g += step;
        }
        keep[keep_word(b, kt, w, c, nkt, nw)] = bits;
    }
}

}  // namespace

cudaError_t launch_keep_fill(const DropParams &d, int bh, int S, uint32_t *keep, cudaStream_t st)
{
    const int nkt = keep_key_tiles(S), nw = keep_row_words(S);
    const bool large = (long long)bh * nkt * nkt >= 40000;
    if (large)
        keep_fill_kernel<4><<<dim3((unsigned)(bh * nkt), (unsigned)((nkt + 3) / 4)), dim3(128, 4), 0, st>>>(
            keep, S, nkt, nw, d.seed, d.keep_thr);
    else
        keep_fill_kernel<1><<<dim3((unsigned)(bh * nkt), (unsigned)nkt), dim3(128, 4), 0, st>>>(keep, S, nkt, nw, d.seed,
                                                                                             d.keep_thr);
    return cudaGetLastError();
}

}  // namespace xfa
