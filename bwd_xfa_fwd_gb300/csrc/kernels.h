// Internal launcher interface between the C-ABI front end (xfa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "xfa.h"

namespace xfa {

// Dropout on the attention probabilities (see dropout.cuh): element (b, i, j) of the
// [bh, S, S] probabilities is kept when the 24-bit draw of its flat index is >= keep_thr
// (= ceil(p * 2^24), so the test equals u = draw / 2^24 >= p exactly) and then scaled by
// inv_keep = 1 / (1 - p).  on == false: no dropout (the plain kernels run).
// keep_out / keep_in: the decisions cached as bits between the forward and the backward (the
// tensor-core bf16 kernels only; see keep_word in dropout.cuh for the layout): the forward also
// writes every decision it draws to keep_out, the backward reads them from keep_in instead of
// drawing them again.  keep_nkt / keep_w: key tiles and query-row words of that layout.
struct DropParams {
    bool on = false;
    uint32_t keep_thr = 0;
    float inv_keep = 1.0f;
    float keep_frac = 1.0f;   // 1 - p
    uint64_t seed = 0;
    uint32_t *keep_out = nullptr;
    const uint32_t *keep_in = nullptr;
    int keep_nkt = 0, keep_w = 0;
};

// Key tiles (128 keys) and query-row words (32 rows, four per 128-row query tile) of the cached
// keep bits of a [bh, S, S] probability tensor.
inline int keep_key_tiles(int S) { return (S + 127) / 128; }
inline int keep_row_words(int S) { return 4 * keep_key_tiles(S); }
inline size_t keep_bits_bytes(int bh, int S)
{
    return (size_t)bh * (size_t)keep_key_tiles(S) * (size_t)keep_row_words(S) * 128u * 4u;
}

struct FwdParams {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int bh, S, hd;
    float scale;
    int dtype;
    int *status;   // device status word
    DropParams drop;
};

struct BwdParams {
    const void *q, *k, *v, *out, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int bh, S, hd;
    float scale;
    int dtype;
    // workspace views
    float *D;       // [bh][S_pad]  D_i = dO_i . O_i (0 on padded rows)
    float *Lg;      // [bh][S_pad]  -L_i * log2(e) (-inf on padded rows)
    float *dq_acc;  // [bh][S][hd]  fp32 dQ accumulator (== dq when dtype is fp32)
    int S_pad;
    float lg_bias = 0.0f;   // added to Lg by the pre-pass (log2(1 / (1 - p)) for the tcgen05 dropout backward)
    int *status;
    DropParams drop;
};

// Rows of D / Lg are padded to a multiple of this.
constexpr int kRowPad = 128;

// Heads a tensor-core kernel schedules together.  Long sequences go in bundles of `dflt`
// heads, longest work first within a bundle, so that the operands of the heads in flight stay
// in L2; when four [bh, S, hd] operands fit in 64 MiB (a fraction of the 129 MB L2) the whole
// grid is one bundle, i.e. longest work first across all heads, which packs the waves of a
// short-sequence grid best.
inline int head_bundle(int bh, int S, int hd, int elt_bytes, int dflt)
{
    const double bytes = 4.0 * (double)bh * (double)S * (double)hd * (double)elt_bytes;
    return bytes <= 64.0 * 1024.0 * 1024.0 ? bh : dflt;
}

// SIMT (FFMA) family: any dtype, hd in {32, 64, 128}.
cudaError_t launch_simt_fwd(const FwdParams &p, cudaStream_t st);
cudaError_t launch_simt_bwd(const BwdParams &p, cudaStream_t st);

// Backward pre-pass: D = rowdot(dO, O), Lg = -lse * log2(e), padded rows filled.
cudaError_t launch_bwd_prep(const BwdParams &p, cudaStream_t st);
// Plain rowdot into an unpadded [bh][S] array.
cudaError_t launch_rowdot(const void *out, const void *dout, float *d, int bh, int S, int hd, int dtype,
                          cudaStream_t st);
// dq (dtype) = dq_acc (fp32), n elements.
cudaError_t launch_convert_dq(const float *acc, void *dq, size_t n, int dtype, cudaStream_t st);
// dst += src, n elements of dtype.
cudaError_t launch_accumulate(void *dst, const void *src, size_t n, int dtype, cudaStream_t st);
// Every cached keep bit at or below the diagonal blocks (keep_word layout) drawn from d.seed.
cudaError_t launch_keep_fill(const DropParams &d, int bh, int S, uint32_t *keep, cudaStream_t st);
// A kernel waiting on a barrier nothing arrives on, for at most timeout_us.
cudaError_t launch_selftest_timeout(unsigned timeout_us, int *status, cudaStream_t st);

// tcgen05 family: bf16, hd in {64, 128}.  Return an XFA_* code.
int launch_tc_fwd(const FwdParams &p, cudaStream_t st);
// Key-tile backward: dK, dV and, when fused_dq, dQ summed into p.dq_acc.
int launch_tc_bwd(const BwdParams &p, cudaStream_t st, bool fused_dq);
// Query-tile dQ pass: writes p.dq (bf16) directly, no atomics.
int launch_tc_dq(const BwdParams &p, cudaStream_t st);

// 3xTF32 tensor-core family: fp32, hd in {32, 64}.  Return an XFA_* code.
int launch_tf_fwd(const FwdParams &p, cudaStream_t st);
// dK, dV by key tiles, then dQ by query tiles (no atomics); writes p.dq / p.dk / p.dv.
int launch_tf_bwd(const BwdParams &p, cudaStream_t st);

// Streaming multiprocessors of the current device (queried once per device), for persistent grids.
int device_sm_count();

// Work-item counter slots of a persistent kernel (two words each: items claimed, CTAs finished).
// Launches take slots round-robin so that launches in flight on different streams use different
// slots; each launch's last CTA sets its slot back to zero.  A launch captured into a CUDA graph
// keeps its slot for every replay, so captured launches take theirs from a separate pool: an
// eager launch never shares a slot with a graph's, and graph replays that overlap one another
// share a slot only after kSchedCapturedSlots captures of the same kernel.
constexpr unsigned kSchedEagerSlots = 64;
constexpr unsigned kSchedCapturedSlots = 448;
constexpr unsigned kSchedSlots = kSchedEagerSlots + kSchedCapturedSlots;
struct SchedSlots {
    std::atomic<unsigned> eager{0};
    std::atomic<unsigned> captured{0};
};
// The slot (index into a kernel's [2 * kSchedSlots] counter array) of a launch on `st`;
// XFA_OK or an error code (a failed capture-status query).
int sched_slot(cudaStream_t st, SchedSlots &slots, unsigned *slot);

// Encodes the TMA descriptors; resolved once from the driver (xfa_api.cu).
int encode_tmap_bf16_3d(void *tmap, const void *base, int hd, int S, int bh, int box_rows);

}  // namespace xfa
