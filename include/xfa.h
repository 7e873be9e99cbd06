/*
 * xfa.h -- C ABI of libxfa.so: fused causal flash-attention, forward and
 * backward, for NVIDIA GB300 (sm_103a).
 *
 * The operation is causal scaled-dot-product attention as defined in
 * "xtrain docs/13-flash-attention.md", section "什么是 flash-attention":
 *
 *   s_ij = scale * Q_i . K_j           for key j <= query i (j > i is masked)
 *   P_ij = softmax_j(s_ij)             row-wise over the unmasked keys
 *   O_i  = sum_j P_ij V_j
 *   L_i  = m_i + ln(l_i) = ln sum_j exp(s_ij)     (natural-log logsumexp)
 *
 * and its gradients through the same page's flash backward
 * (D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i) scale,  dP_ij = dO_i . V_j):
 *
 *   dQ_i = sum_j dS_ij K_j,   dK_j = sum_i dS_ij Q_i,   dV_j = sum_i P_ij dO_i.
 *
 * Conventions shared by every entry point:
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are contiguous row-major [bh][S][hd]
 *     arrays in device memory, element type given by `dtype` (xfa_dtype).
 *     bh = batch * heads; every head is an independent problem.  The query
 *     position used by the causal mask is the row index within S (the
 *     "i % S" of the page's flattened [B*S] rows).
 *   - lse is a contiguous [bh][S] fp32 device array (natural log).
 *   - Pointers must be 16-byte aligned device pointers and must not alias
 *     each other (inputs may alias inputs).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on `stream` and returns; it never synchronises,
 *     allocates or frees memory.  The caller owns every buffer.
 *   - Supported shapes: bh >= 1, S >= 1 (any S: ragged tails are masked),
 *     hd in {32, 64, 128}; bh * S * hd < 2^31.  scale must be finite and > 0.
 *   - Return value: XFA_OK, or an error code.  Argument errors are detected
 *     on the host before anything is enqueued, and nothing is written.
 *     A CUDA launch error is returned as XFA_ERR_CUDA_BASE + cudaError_t.
 *     A kernel that gives up waiting on its own pipeline (see xfa_last_status)
 *     leaves its outputs undefined.
 */
#ifndef XFA_H
#define XFA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V, O, dO, dQ, dK, dV.  Arithmetic is fp32 throughout
 * (fp32 accumulation; bf16 operands feed the tensor cores). */
typedef enum { XFA_F32 = 0, XFA_BF16 = 1 } xfa_dtype;

/* Kernel family selector for the *_impl entry points. */
typedef enum {
    XFA_IMPL_AUTO = 0,        /* the fastest tcgen05 variant where supported, else SIMT */
    XFA_IMPL_SIMT = 1,        /* fp32 FFMA tiled kernels (every dtype and hd) */
    XFA_IMPL_TCGEN05 = 2,     /* tcgen05.mma + TMEM kernels.  bf16, hd in {64, 128}: TMA-fed
                                 kernels whose backward sums dQ over key tiles with fp32
                                 reductions, so dQ may differ in the last bits from run to run.
                                 fp32, hd in {32, 64}: the 3xTF32 kernels (each operand split
                                 into two tf32 parts, three MMAs per product, about 2^-21
                                 relative error per product); their backward forms dQ in a
                                 query-tile pass without atomics, so results are bit-reproducible */
    XFA_IMPL_TCGEN05_DET = 3  /* as XFA_IMPL_TCGEN05, but the bf16 backward also forms dQ in a
                                 separate query-tile pass without atomics: bit-reproducible
                                 results (fp32: the same kernels as XFA_IMPL_TCGEN05) */
} xfa_impl;

enum {
    XFA_OK = 0,
    XFA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale */
    XFA_ERR_UNSUPPORTED = 2,  /* valid but unsupported combination (hd, dtype, impl) */
    XFA_ERR_TIMEOUT = 3,      /* a kernel gave up waiting on its pipeline (xfa_last_status) */
    XFA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than xfa_bwd_workspace_bytes */
    XFA_ERR_DEVICE = 5,       /* no usable device, or not an sm_103 device for tcgen05 */
    XFA_ERR_CUDA_BASE = 1000  /* + cudaError_t of a failed CUDA runtime call */
};

/*
 * Forward.  Passage: "xtrain docs/13-flash-attention.md", section
 * "什么是 flash-attention" (online-softmax recurrence over KV tiles with running
 * max m, running sum l and an [hd] accumulator; out = acc / l; L = m + log l;
 * tiles wholly above the diagonal skipped) and design decision ② (only the
 * O(N) logsumexp is kept for the backward).
 *   q, k, v : [bh][S][hd] inputs (dtype)
 *   out     : [bh][S][hd] output O (dtype), overwritten
 *   lse     : [bh][S] fp32 output L (natural log), overwritten
 */
int xfa_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
            int bh, int S, int hd, float scale, int dtype, void *stream);

/* xfa_fwd with an explicit kernel family (xfa_impl). */
int xfa_fwd_impl(const void *q, const void *k, const void *v, void *out, float *lse,
                 int bh, int S, int hd, float scale, int dtype, int impl, void *stream);

/*
 * Bytes of device workspace xfa_bwd needs for this shape (a pure function of
 * its arguments; 0 for invalid arguments).  Holds D [bh][S'] and -L*log2(e)
 * [bh][S'] fp32 (S' = S rounded up to 128) and, for bf16, an fp32 dQ
 * accumulator [bh][S][hd].
 */
size_t xfa_bwd_workspace_bytes(int bh, int S, int hd, int dtype);

/*
 * Backward.  Passage: "xtrain docs/13-flash-attention.md", section
 * "什么是 flash-attention" (recompute s_ij and p_ij = exp(s_ij - L_i) from Q, K
 * and L; dp_ij = dO_i . V_j; ds_ij = p_ij (dp_ij - D_i) scale; dQ, dK, dV
 * accumulation) and design decision ③ (D_i = sum_d dO_i[d] O_i[d] computed in
 * one pass first).
 *   q, k, v      : forward inputs (dtype)
 *   out, lse     : forward outputs O (dtype) and L (fp32) of the same call
 *   dout         : [bh][S][hd] upstream gradient dO (dtype)
 *   dq, dk, dv   : [bh][S][hd] gradients (dtype), OVERWRITTEN (not accumulated;
 *                  fan-out accumulation is the caller's, e.g. xfa_accumulate)
 *   workspace    : device scratch of at least xfa_bwd_workspace_bytes() bytes,
 *                  16-byte aligned; contents on entry are ignored
 * Enqueues, in order on `stream`: the D pre-pass, the backward kernel and,
 * for bf16, the dQ fp32 -> bf16 conversion.
 */
int xfa_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
            const float *lse, void *dq, void *dk, void *dv,
            int bh, int S, int hd, float scale, int dtype,
            void *workspace, size_t workspace_bytes, void *stream);

/* xfa_bwd with an explicit kernel family (xfa_impl). */
int xfa_bwd_impl(const void *q, const void *k, const void *v, const void *out, const void *dout,
                 const float *lse, void *dq, void *dk, void *dv,
                 int bh, int S, int hd, float scale, int dtype,
                 void *workspace, size_t workspace_bytes, int impl, void *stream);

/*
 * Forward and backward with dropout on the attention probabilities.  Passage:
 * "xtrain docs/17-dropout.md", section "Key Design Decisions" (counter-based
 * draw: key = seed XOR (idx * 0x9E3779B97F4A7C15), h = splitmix64(key),
 * u = (h >> 40) / 2^24, keep = u >= p; kept elements scaled by 1 / (1 - p);
 * the backward re-draws the same mask from (seed, idx)).  The page applies it to
 * activations and leaves the attention probabilities out; here it sits between
 * the softmax and the product with V:
 *   O_i = sum_j P_ij C_ij V_j,   C_ij = keep(seed, (b*S + i)*S + j) / (1 - p),
 * L is the plain logsumexp (the softmax is unchanged), and the backward uses
 * dP_ij = C_ij dO_i . V_j in place of dO_i . V_j (D_i = dO_i . O_i still holds).
 *   p_drop : rate in [0, 1); anything else (or NaN) gives XFA_ERR_INVALID_ARG.
 *            p_drop == 0 runs the plain kernels (results bit for bit those of
 *            xfa_fwd_impl / xfa_bwd_impl).
 *   seed   : 64-bit seed; the forward and the backward of one use must get the
 *            same seed and p_drop.
 * Other arguments as xfa_fwd_impl / xfa_bwd_impl.  Families: XFA_IMPL_AUTO,
 * XFA_IMPL_TCGEN05 (bf16 with hd 64 / 128, fp32 with hd 32 / 64) and XFA_IMPL_SIMT;
 * XFA_IMPL_TCGEN05_DET with fp32 as XFA_IMPL_TCGEN05; the bf16 backward with
 * XFA_IMPL_TCGEN05_DET and p_drop > 0 returns XFA_ERR_UNSUPPORTED.
 */
int xfa_fwd_dropout(const void *q, const void *k, const void *v, void *out, float *lse,
                    int bh, int S, int hd, float scale, int dtype,
                    float p_drop, unsigned long long seed, int impl, void *stream);

int xfa_bwd_dropout(const void *q, const void *k, const void *v, const void *out, const void *dout,
                    const float *lse, void *dq, void *dk, void *dv,
                    int bh, int S, int hd, float scale, int dtype,
                    float p_drop, unsigned long long seed,
                    void *workspace, size_t workspace_bytes, int impl, void *stream);

/*
 * Dropout with the keep decisions cached in a caller-owned bit buffer.  Passage:
 * "xtrain docs/17-dropout.md", sections "Goal" and "Key Design Decisions" (the mask is
 * generated once from (seed, index) and the forward and the backward both apply that same
 * cached mask).  The draw is bound by the integer multiplier; reading a bit is not.
 *   xfa_dropout_keep_fill  : draws every decision into keep_bits (a kernel of its own, e.g. on
 *                            another stream ahead of the attention).
 *   xfa_fwd_dropout_keep   : xfa_fwd_dropout that also stores every decision it draws.
 *   xfa_fwd_dropout_cached : xfa_fwd_dropout reading the decisions from keep_bits.
 *   xfa_bwd_dropout_cached : xfa_bwd_dropout reading the decisions from keep_bits.
 * The readers take no seed.  Whichever way keep_bits was filled (fill or the storing forward,
 * with the same bh, S, p_drop and seed), results are bit for bit those of the drawing calls.
 *   keep_bits  : device buffer of at least xfa_dropout_keep_bytes(bh, S) bytes, 16-byte
 *                aligned, owned by the caller.  Layout: bit i of 32-bit word
 *                ((b * nkt + kt) * nw + w) * 128 + c is the decision of probability
 *                (b, query row 32 w + i, key 128 kt + c), nkt = ceil(S / 128),
 *                nw = 4 nkt; the writers write the words with w >= 4 kt (the blocks at
 *                or below the diagonal, rows and keys past S included), the rest stay as
 *                they were.
 *   keep_bytes : size of keep_bits in bytes.
 * Families: the tensor-core bf16 kernels (hd 64 / 128; XFA_IMPL_AUTO or XFA_IMPL_TCGEN05,
 * and XFA_IMPL_TCGEN05_DET for the forwards); fp32, the SIMT family or XFA_IMPL_TCGEN05_DET in
 * the backward give XFA_ERR_UNSUPPORTED.  p_drop == 0 runs the plain kernels (the fill does
 * nothing) and leaves keep_bits untouched.  A missing, misaligned or short buffer gives
 * XFA_ERR_INVALID_ARG.
 */
size_t xfa_dropout_keep_bytes(int bh, int S);   /* 0 for bh < 1, S < 1 or a shape no call accepts */

int xfa_dropout_keep_fill(int bh, int S, float p_drop, unsigned long long seed,
                          void *keep_bits, size_t keep_bytes, void *stream);

int xfa_fwd_dropout_keep(const void *q, const void *k, const void *v, void *out, float *lse,
                         int bh, int S, int hd, float scale, int dtype,
                         float p_drop, unsigned long long seed,
                         void *keep_bits, size_t keep_bytes, int impl, void *stream);

int xfa_fwd_dropout_cached(const void *q, const void *k, const void *v, void *out, float *lse,
                           int bh, int S, int hd, float scale, int dtype, float p_drop,
                           const void *keep_bits, size_t keep_bytes, int impl, void *stream);

int xfa_bwd_dropout_cached(const void *q, const void *k, const void *v, const void *out, const void *dout,
                           const float *lse, void *dq, void *dk, void *dv,
                           int bh, int S, int hd, float scale, int dtype, float p_drop,
                           const void *keep_bits, size_t keep_bytes,
                           void *workspace, size_t workspace_bytes, int impl, void *stream);

/*
 * The three stages of xfa_bwd as separate calls, for callers that schedule
 * (or time) them individually.  xfa_bwd_impl is exactly prep, main, finish
 * in this order on one stream, with the same arguments and workspace.
 *   prep   : D_i = dO_i . O_i and -L_i * log2(e) into the workspace (padded
 *            rows: D = 0, -L*log2(e) = -inf), and clears the fp32 dQ accumulator (the
 *            workspace for bf16, dq itself for fp32) when the implementation uses one.
 *   main   : the backward kernels: dK, dV written; dQ summed into the accumulator,
 *            or (XFA_IMPL_TCGEN05_DET) written directly by the query-tile dQ pass.
 *   finish : dQ accumulator -> dq in the output dtype (nothing to do for fp32 or
 *            for XFA_IMPL_TCGEN05_DET).
 * `impl` must be the same for the three stages of one backward.
 * Same argument rules and error codes as xfa_bwd.
 */
int xfa_bwd_prep(const void *out, const void *dout, const float *lse, void *dq, int bh, int S, int hd, int dtype,
                 void *workspace, size_t workspace_bytes, int impl, void *stream);
int xfa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk, void *dv,
                 int bh, int S, int hd, float scale, int dtype, void *workspace, size_t workspace_bytes, int impl,
                 void *stream);
int xfa_bwd_finish(void *dq, int bh, int S, int hd, int dtype, void *workspace, size_t workspace_bytes,
                   int impl, void *stream);

/*
 * Size in bytes of the fixed device scratch array used by xfa_bwd_noalloc.
 * It covers xfa_bwd_workspace_bytes() up to 32 MiB, i.e. bf16 bh*S*hd up to
 * about 8 million elements at hd = 128 (bh = 32, S = 1024 needs 16.25 MiB).
 */
#define XFA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * xfa_bwd for callers that cannot allocate device memory when they run the
 * backward (a host framework that has reserved the device memory for its own
 * allocator, a plug-in host that forbids allocation in its callbacks, code
 * that cannot take cudaMalloc's implicit device synchronisation).  The pages
 * have no counterpart: this is a deployment variant of xfa_bwd, not part of
 * the method.
 *   Arguments as xfa_bwd, without the workspace: the scratch is one
 *   file-scope device array of XFA_NOALLOC_SCRATCH_BYTES inside the library,
 *   kept on a device until the process exits.
 *   Returns XFA_ERR_WORKSPACE when xfa_bwd_workspace_bytes() for the shape
 *   exceeds XFA_NOALLOC_SCRATCH_BYTES; otherwise as xfa_bwd.
 *   The entry point itself calls no cudaMalloc/cudaFree or allocating library
 *   routine.  The array sits in a module of the library that CUDA loads on
 *   first use (lazy module loading, CUDA's default): the first call on each
 *   device, made with that device current, loads that module -- which
 *   reserves the XFA_NOALLOC_SCRATCH_BYTES on the device and may synchronise
 *   it -- and resolves the array's device address (cudaGetSymbolAddress).  That
 *   first call can therefore fail with XFA_ERR_CUDA_BASE +
 *   cudaErrorMemoryAllocation when the device is already full; make it at
 *   set-up time (a small problem will do), before any stream capture and
 *   outside callbacks that forbid allocation.  Later calls on that device
 *   allocate nothing.  (With CUDA_MODULE_LOADING=EAGER the module, and the
 *   array, are loaded with the library when the context is created.)
 *   Every call shares the array and it keeps the last call's contents (each
 *   call rewrites or clears everything it reads before reading it); calls
 *   that overlap on the GPU race on it.
 */
int xfa_bwd_noalloc(const void *q, const void *k, const void *v, const void *out, const void *dout,
                    const float *lse, void *dq, void *dk, void *dv,
                    int bh, int S, int hd, float scale, int dtype, void *stream);

/*
 * The backward's pre-pass on its own: D[b][i] = sum_d dout[b][i][d] * out[b][i][d]
 * with fp32 accumulation.  Passage: "xtrain docs/13-flash-attention.md",
 * design decision ③ (D_i = sum_d dO_i[d] O_i[d]).
 *   out, dout : [bh][S][hd] (dtype);  d : [bh][S] fp32 output, overwritten.
 */
int xfa_rowdot(const void *out, const void *dout, float *d, int bh, int S, int hd, int dtype, void *stream);

/*
 * dst[i] += src[i] for i < n (dtype elements, fp32 arithmetic).  The tape's
 * fan-out gradient accumulation: "xtrain docs/03-autograd-engine.md", section
 * "梯度累加（扇出求和）" (every push_grad sums into the existing gradient).
 * dst and src must not overlap partially.
 */
int xfa_accumulate(void *dst, const void *src, size_t n, int dtype, void *stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns XFA_OK, XFA_ERR_TIMEOUT when a kernel
 * since the last call gave up on a pipeline wait (every wait in every kernel
 * has a time limit of about one second, after which the kernel records the
 * timeout, drains its own in-flight copies, frees its tensor memory and
 * exits), or XFA_ERR_CUDA_BASE + a CUDA error.  The pages' own kernels
 * synchronise after every operation ("xtrain docs/03-autograd-engine.md",
 * section "kernel 实现要点"); here that check is this one explicit call.
 */
int xfa_last_status(void *stream);

/* The same call under its earlier name (kept for existing callers). */
int xfa_status(void *stream);

/*
 * Self-test of the timeout path: enqueues one single-CTA kernel that waits on
 * a shared-memory barrier which nothing ever arrives on, with a limit of
 * `timeout_us` microseconds (1 .. 1000000).  The kernel then records
 * XFA_ERR_TIMEOUT in the status word and returns; read it with xfa_last_status.
 * No counterpart on the pages: it exists so the timeout path can be tested
 * without hanging a GPU.
 */
int xfa_selftest_timeout(unsigned timeout_us, void *stream);

/* Static description of an error code. */
const char *xfa_strerror(int code);

/* ABI version (major * 100 + minor). */
int xfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* XFA_H */
