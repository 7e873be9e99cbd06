// C-ABI front end of libxfa.so (declared in include/xfa.h): argument
// validation, workspace layout, TMA descriptor encoding, kernel-family
// dispatch and the device status word.  Nothing here allocates, frees or
// synchronises except xfa_last_status (and its older name xfa_status), which is
// documented to synchronise.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "xfa.h"

namespace xfa {

// Library status word: kernels record XFA_ERR_TIMEOUT here (first error wins).
__device__ int g_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];
int g_is_sm103[kMaxDevices];   // 0 unknown, 1 yes, 2 no
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_code(cudaError_t e) { return e == cudaSuccess ? XFA_OK : XFA_ERR_CUDA_BASE + (int)e; }

int current_device(int *dev)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_code(e);
    if (*dev < 0 || *dev >= kMaxDevices) return XFA_ERR_DEVICE;
    return XFA_OK;
}

// Device address of g_status on the current device (resolved once per device).
int status_ptr(int **out)
{
    int dev;
    int rc = current_device(&dev);
    if (rc != XFA_OK) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_status);
        if (e != cudaSuccess) return cuda_code(e);
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return XFA_OK;
}

bool device_is_sm103()
{
    int dev;
    if (current_device(&dev) != XFA_OK) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_is_sm103[dev] == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_is_sm103[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return g_is_sm103[dev] == 1;
}

int g_sm_count[kMaxDevices];   // 0 unknown

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_shape(int bh, int S, int hd, float scale, int dtype)
{
    if (dtype != XFA_F32 && dtype != XFA_BF16) return XFA_ERR_INVALID_ARG;
    if (bh < 1 || S < 1) return XFA_ERR_INVALID_ARG;
    if (hd != 32 && hd != 64 && hd != 128) return XFA_ERR_UNSUPPORTED;
    if ((long long)bh * (long long)S * (long long)hd >= (1ll << 31)) return XFA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return XFA_ERR_INVALID_ARG;
    return XFA_OK;
}

bool tc_supported(int hd, int dtype) { return dtype == XFA_BF16 && (hd == 64 || hd == 128); }

// fp32 on the tensor cores (3xTF32): hd 32 and 64 (hd 128 fp32 tiles do not fit shared memory).
bool tf_supported(int hd, int dtype) { return dtype == XFA_F32 && (hd == 32 || hd == 64); }

enum class Family { Simt, TcFused, TcDet, Tf32 };

// The tcgen05 backward variant XFA_IMPL_AUTO resolves to.
constexpr Family kAutoTc = Family::TcFused;

// Resolve the implementation for a call; XFA_OK and *fam set on success.
int choose_impl(int impl, int hd, int dtype, Family *fam)
{
    switch (impl) {
    case XFA_IMPL_SIMT: *fam = Family::Simt; return XFA_OK;
    case XFA_IMPL_TCGEN05:
    case XFA_IMPL_TCGEN05_DET:
        if (tf_supported(hd, dtype)) {
            if (!device_is_sm103()) return XFA_ERR_DEVICE;
            *fam = Family::Tf32;   // one kernel family for fp32, deterministic by construction
            return XFA_OK;
        }
        if (!tc_supported(hd, dtype)) return XFA_ERR_UNSUPPORTED;
        if (!device_is_sm103()) return XFA_ERR_DEVICE;
        *fam = impl == XFA_IMPL_TCGEN05 ? Family::TcFused : Family::TcDet;
        return XFA_OK;
    case XFA_IMPL_AUTO:
        if (!device_is_sm103()) *fam = Family::Simt;
        else if (tc_supported(hd, dtype)) *fam = kAutoTc;
        else if (tf_supported(hd, dtype)) *fam = Family::Tf32;
        else *fam = Family::Simt;
        return XFA_OK;
    default: return XFA_ERR_INVALID_ARG;
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t off_D, off_Lg, off_dq, total;
    int S_pad;
};

WsLayout ws_layout(int bh, int S, int hd, int dtype)
{
    WsLayout w;
    w.S_pad = (S + kRowPad - 1) / kRowPad * kRowPad;
    const size_t rows = (size_t)bh * (size_t)w.S_pad * sizeof(float);
    w.off_D = 0;
    w.off_Lg = align256(rows);
    w.off_dq = align256(w.off_Lg + rows);
    w.total = w.off_dq + (dtype == XFA_BF16 ? (size_t)bh * S * hd * sizeof(float) : 0);
    return w;
}

int resolve_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return XFA_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_code(e);
    if (q != cudaDriverEntryPointSuccess || !fn) return XFA_ERR_DEVICE;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return XFA_OK;
}

}  // namespace

int device_sm_count()
{
    int dev;
    if (current_device(&dev) != XFA_OK) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int sched_slot(cudaStream_t st, SchedSlots &slots, unsigned *slot)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_code(e);
    if (cs == cudaStreamCaptureStatusActive)
        *slot = kSchedEagerSlots + slots.captured.fetch_add(1u) % kSchedCapturedSlots;
    else
        *slot = slots.eager.fetch_add(1u) % kSchedEagerSlots;
    return XFA_OK;
}

// [bh][S][hd] bf16 tensor as a 3-D TMA map with boxes of 64 columns x box_rows rows,
// 128-byte swizzle; rows past S read as zero.
int encode_tmap_bf16_3d(void *tmap, const void *base, int hd, int S, int bh, int box_rows)
{
    int rc = resolve_encoder();
    if (rc != XFA_OK) return rc;
    const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)S, (cuuint64_t)bh};
    const cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)S * hd * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(static_cast<CUtensorMap *>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? XFA_OK : XFA_ERR_INVALID_ARG;
}

}  // namespace xfa

using namespace xfa;

extern "C" {

int xfa_version(void) { return 100; }

const char *xfa_strerror(int code)
{
    switch (code) {
    case XFA_OK: return "ok";
    case XFA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or scale)";
    case XFA_ERR_UNSUPPORTED: return "unsupported combination of head dim, dtype and kernel family";
    case XFA_ERR_TIMEOUT: return "a kernel gave up waiting on its pipeline (timeout)";
    case XFA_ERR_WORKSPACE: return "workspace missing or too small";
    case XFA_ERR_DEVICE: return "no usable sm_103 device";
    default: break;
    }
    if (code >= XFA_ERR_CUDA_BASE) return cudaGetErrorString((cudaError_t)(code - XFA_ERR_CUDA_BASE));
    return "unknown error";
}

}  // extern "C"

// Dropout parameters of a call: rate p in [0, 1) (NaN rejected); p == 0 leaves dropout off.
static int make_drop(float p, unsigned long long seed, DropParams *d)
{
    if (!(p >= 0.0f && p < 1.0f)) return XFA_ERR_INVALID_ARG;
    *d = DropParams{};
    if (p == 0.0f) return XFA_OK;
    d->on = true;
    d->keep_thr = (uint32_t)ceil((double)p * 16777216.0);   // u = draw / 2^24 >= p  <=>  draw >= keep_thr
    d->inv_keep = (float)(1.0 / (1.0 - (double)p));
    d->keep_frac = (float)(1.0 - (double)p);
    d->seed = seed;
    return XFA_OK;
}

// The cached keep-bit buffer of a dropout call (see DropParams): present, 16-byte aligned and at
// least xfa_dropout_keep_bytes(bh, S) long; sets the layout sizes.
static int keep_args(int bh, int S, const void *keep, size_t keep_bytes, DropParams *d)
{
    if (bh < 1 || S < 1 || (long long)bh * (long long)S >= (1ll << 26)) return XFA_ERR_INVALID_ARG;
    if (!keep || !aligned16(keep) || keep_bytes < keep_bits_bytes(bh, S)) return XFA_ERR_INVALID_ARG;
    d->keep_nkt = keep_key_tiles(S);
    d->keep_w = keep_row_words(S);
    return XFA_OK;
}

static int fwd_run(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S, int hd,
                   float scale, int dtype, const DropParams &drop, int impl, void *stream)
{
    int rc = validate_shape(bh, S, hd, scale, dtype);
    if (rc != XFA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return XFA_ERR_INVALID_ARG;
    Family fam;
    if ((rc = choose_impl(impl, hd, dtype, &fam)) != XFA_OK) return rc;
    // cached keep bits: the tensor-core bf16 kernels only
    if ((drop.keep_out || drop.keep_in) && fam != Family::TcFused && fam != Family::TcDet) return XFA_ERR_UNSUPPORTED;
    FwdParams p{q, k, v, out, lse, bh, S, hd, scale, dtype, nullptr};
    p.drop = drop;
    if ((rc = status_ptr(&p.status)) != XFA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (fam == Family::Tf32) return launch_tf_fwd(p, st);
    if (fam != Family::Simt) return launch_tc_fwd(p, st);
    return cuda_code(launch_simt_fwd(p, st));
}

extern "C" {

int xfa_fwd_impl(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S, int hd,
                 float scale, int dtype, int impl, void *stream)
{
    return fwd_run(q, k, v, out, lse, bh, S, hd, scale, dtype, DropParams{}, impl, stream);
}

int xfa_fwd_dropout(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S, int hd,
                    float scale, int dtype, float p_drop, unsigned long long seed, int impl, void *stream)
{
    DropParams d;
    const int rc = make_drop(p_drop, seed, &d);
    if (rc != XFA_OK) return rc;
    return fwd_run(q, k, v, out, lse, bh, S, hd, scale, dtype, d, impl, stream);
}

size_t xfa_dropout_keep_bytes(int bh, int S)
{
    if (bh < 1 || S < 1 || (long long)bh * (long long)S >= (1ll << 26)) return 0;
    return keep_bits_bytes(bh, S);
}

int xfa_fwd_dropout_keep(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S, int hd,
                         float scale, int dtype, float p_drop, unsigned long long seed, void *keep_bits,
                         size_t keep_bytes, int impl, void *stream)
{
    DropParams d;
    int rc = make_drop(p_drop, seed, &d);
    if (rc != XFA_OK || (rc = keep_args(bh, S, keep_bits, keep_bytes, &d)) != XFA_OK) return rc;
    if (d.on) d.keep_out = static_cast<uint32_t *>(keep_bits);
    return fwd_run(q, k, v, out, lse, bh, S, hd, scale, dtype, d, impl, stream);
}

int xfa_fwd_dropout_cached(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S,
                           int hd, float scale, int dtype, float p_drop, const void *keep_bits, size_t keep_bytes,
                           int impl, void *stream)
{
    DropParams d;
    int rc = make_drop(p_drop, 0, &d);
    if (rc != XFA_OK || (rc = keep_args(bh, S, keep_bits, keep_bytes, &d)) != XFA_OK) return rc;
    if (d.on) d.keep_in = static_cast<const uint32_t *>(keep_bits);
    return fwd_run(q, k, v, out, lse, bh, S, hd, scale, dtype, d, impl, stream);
}

int xfa_dropout_keep_fill(int bh, int S, float p_drop, unsigned long long seed, void *keep_bits, size_t keep_bytes,
                          void *stream)
{
    DropParams d;
    int rc = make_drop(p_drop, seed, &d);
    if (rc != XFA_OK || (rc = keep_args(bh, S, keep_bits, keep_bytes, &d)) != XFA_OK) return rc;
    if (!d.on) return XFA_OK;   // p_drop == 0: the consumers run the plain kernels and read nothing
    if (!device_is_sm103()) return XFA_ERR_DEVICE;
    return cuda_code(launch_keep_fill(d, bh, S, static_cast<uint32_t *>(keep_bits), static_cast<cudaStream_t>(stream)));
}

int xfa_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int bh, int S, int hd, float scale,
            int dtype, void *stream)
{
    return xfa_fwd_impl(q, k, v, out, lse, bh, S, hd, scale, dtype, XFA_IMPL_AUTO, stream);
}

size_t xfa_bwd_workspace_bytes(int bh, int S, int hd, int dtype)
{
    if (validate_shape(bh, S, hd, 1.0f, dtype) != XFA_OK) return 0;
    return ws_layout(bh, S, hd, dtype).total;
}

// Validates the arguments every backward stage shares and fills the params.
static int bwd_setup(BwdParams &p, const void *q, const void *k, const void *v, const void *out, const void *dout,
                     const float *lse, void *dq, void *dk, void *dv, int bh, int S, int hd, float scale, int dtype,
                     void *workspace, size_t workspace_bytes)
{
    int rc = validate_shape(bh, S, hd, scale, dtype);
    if (rc != XFA_OK) return rc;
    const void *ptrs[] = {q, k, v, out, dout, lse, dq, dk, dv};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return XFA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(bh, S, hd, dtype);
    if (!aligned16(workspace) || workspace_bytes < w.total) return XFA_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p = BwdParams{};
    p.q = q; p.k = k; p.v = v; p.out = out; p.dout = dout; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.bh = bh; p.S = S; p.hd = hd; p.scale = scale; p.dtype = dtype;
    p.D = reinterpret_cast<float *>(ws + w.off_D);
    p.Lg = reinterpret_cast<float *>(ws + w.off_Lg);
    p.dq_acc = dtype == XFA_BF16 ? reinterpret_cast<float *>(ws + w.off_dq) : static_cast<float *>(dq);
    p.S_pad = w.S_pad;
    return status_ptr(&p.status);
}

// Any 16-byte aligned non-null placeholder for pointers a stage does not touch.
static const void *unused_ptr(const void *p) { return p; }

// The three stages of one backward for the resolved family.
static int stage_prep(BwdParams p, Family fam, cudaStream_t st)
{
    if (fam == Family::TcDet || fam == Family::Tf32) p.dq_acc = nullptr;   // no accumulator to clear
    return cuda_code(launch_bwd_prep(p, st));
}

static int stage_main(const BwdParams &p, Family fam, cudaStream_t st)
{
    switch (fam) {
    case Family::Simt: return cuda_code(launch_simt_bwd(p, st));
    case Family::TcFused: return launch_tc_bwd(p, st, true);
    case Family::TcDet: {
        int rc = launch_tc_bwd(p, st, false);
        return rc == XFA_OK ? launch_tc_dq(p, st) : rc;
    }
    case Family::Tf32: return launch_tf_bwd(p, st);
    }
    return XFA_ERR_INVALID_ARG;
}

static int stage_finish(const BwdParams &p, Family fam, cudaStream_t st)
{
    if (p.dtype != XFA_BF16 || fam == Family::TcDet) return XFA_OK;
    return cuda_code(launch_convert_dq(p.dq_acc, p.dq, (size_t)p.bh * p.S * p.hd, p.dtype, st));
}

int xfa_bwd_prep(const void *out, const void *dout, const float *lse, void *dq, int bh, int S, int hd, int dtype,
                 void *workspace, size_t workspace_bytes, int impl, void *stream)
{
    BwdParams p;
    const void *u = unused_ptr(out);
    int rc = bwd_setup(p, u, u, u, out, dout, lse, dq, const_cast<void *>(u), const_cast<void *>(u), bh, S, hd,
                       1.0f, dtype, workspace, workspace_bytes);
    if (rc != XFA_OK) return rc;
    Family fam;
    if ((rc = choose_impl(impl, hd, dtype, &fam)) != XFA_OK) return rc;
    return stage_prep(p, fam, static_cast<cudaStream_t>(stream));
}

int xfa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk, void *dv, int bh,
                 int S, int hd, float scale, int dtype, void *workspace, size_t workspace_bytes, int impl,
                 void *stream)
{
    BwdParams p;
    int rc = bwd_setup(p, q, k, v, dout, dout, reinterpret_cast<const float *>(workspace), dq, dk, dv, bh, S, hd,
                       scale, dtype, workspace, workspace_bytes);
    if (rc != XFA_OK) return rc;
    Family fam;
    if ((rc = choose_impl(impl, hd, dtype, &fam)) != XFA_OK) return rc;
    return stage_main(p, fam, static_cast<cudaStream_t>(stream));
}

int xfa_bwd_finish(void *dq, int bh, int S, int hd, int dtype, void *workspace, size_t workspace_bytes, int impl,
                   void *stream)
{
    BwdParams p;
    int rc = bwd_setup(p, dq, dq, dq, dq, dq, reinterpret_cast<const float *>(workspace), dq, dq, dq, bh, S, hd, 1.0f,
                       dtype, workspace, workspace_bytes);
    if (rc != XFA_OK) return rc;
    Family fam;
    if ((rc = choose_impl(impl, hd, dtype, &fam)) != XFA_OK) return rc;
    return stage_finish(p, fam, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

static int bwd_run(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                   void *dq, void *dk, void *dv, int bh, int S, int hd, float scale, int dtype, void *workspace,
                   size_t workspace_bytes, const DropParams &drop, int impl, void *stream)
{
    BwdParams p;
    int rc = bwd_setup(p, q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, workspace, workspace_bytes);
    if (rc != XFA_OK) return rc;
    p.drop = drop;
    Family fam;
    if ((rc = choose_impl(impl, hd, dtype, &fam)) != XFA_OK) return rc;
    if (drop.on && fam == Family::TcDet) return XFA_ERR_UNSUPPORTED;   // dropout: every family but bf16 TcDet
    if (drop.keep_in && fam != Family::TcFused) return XFA_ERR_UNSUPPORTED;   // cached keep bits: bf16 tcgen05
    // the tcgen05 dropout backward takes P / (1 - p) straight from the exponential: 2^(s c - L log2 e + log2(1 / (1 - p)))
    if (drop.on && fam == Family::TcFused) p.lg_bias = (float)std::log2((double)drop.inv_keep);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = stage_prep(p, fam, st)) != XFA_OK) return rc;
    if ((rc = stage_main(p, fam, st)) != XFA_OK) return rc;
    return stage_finish(p, fam, st);
}

extern "C" {

int xfa_bwd_impl(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                 void *dq, void *dk, void *dv, int bh, int S, int hd, float scale, int dtype, void *workspace,
                 size_t workspace_bytes, int impl, void *stream)
{
    return bwd_run(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, workspace, workspace_bytes,
                   DropParams{}, impl, stream);
}

int xfa_bwd_dropout(const void *q, const void *k, const void *v, const void *out, const void *dout,
                    const float *lse, void *dq, void *dk, void *dv, int bh, int S, int hd, float scale, int dtype,
                    float p_drop, unsigned long long seed, void *workspace, size_t workspace_bytes, int impl,
                    void *stream)
{
    DropParams d;
    const int rc = make_drop(p_drop, seed, &d);
    if (rc != XFA_OK) return rc;
    return bwd_run(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, workspace, workspace_bytes, d, impl,
                   stream);
}

int xfa_bwd_dropout_cached(const void *q, const void *k, const void *v, const void *out, const void *dout,
                         const float *lse, void *dq, void *dk, void *dv, int bh, int S, int hd, float scale,
                         int dtype, float p_drop, const void *keep_bits, size_t keep_bytes, void *workspace,
                         size_t workspace_bytes, int impl, void *stream)
{
    DropParams d;
    int rc = make_drop(p_drop, 0, &d);
    if (rc != XFA_OK || (rc = keep_args(bh, S, keep_bits, keep_bytes, &d)) != XFA_OK) return rc;
    if (d.on) d.keep_in = static_cast<const uint32_t *>(keep_bits);
    return bwd_run(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, workspace, workspace_bytes, d, impl,
                   stream);
}

int xfa_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
            void *dq, void *dk, void *dv, int bh, int S, int hd, float scale, int dtype, void *workspace,
            size_t workspace_bytes, void *stream)
{
    return xfa_bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, workspace, workspace_bytes,
                        XFA_IMPL_AUTO, stream);
}

int xfa_rowdot(const void *out, const void *dout, float *d, int bh, int S, int hd, int dtype, void *stream)
{
    int rc = validate_shape(bh, S, hd, 1.0f, dtype);
    if (rc != XFA_OK) return rc;
    if (!aligned16(out) || !aligned16(dout) || !aligned16(d)) return XFA_ERR_INVALID_ARG;
    return cuda_code(launch_rowdot(out, dout, d, bh, S, hd, dtype, static_cast<cudaStream_t>(stream)));
}

int xfa_accumulate(void *dst, const void *src, size_t n, int dtype, void *stream)
{
    if (dtype != XFA_F32 && dtype != XFA_BF16) return XFA_ERR_INVALID_ARG;
    if (n == 0) return XFA_OK;
    if (!dst || !src) return XFA_ERR_INVALID_ARG;
    return cuda_code(launch_accumulate(dst, src, n, dtype, static_cast<cudaStream_t>(stream)));
}

int xfa_status(void *stream) { return xfa_last_status(stream); }

int xfa_last_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_code(e);
    int *sp = nullptr;
    int rc = status_ptr(&sp);
    if (rc != XFA_OK) return rc;
    int code = 0;
    e = cudaMemcpyFromSymbol(&code, g_status, sizeof(int));
    if (e != cudaSuccess) return cuda_code(e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_code(e);
    return code;
}

int xfa_selftest_timeout(unsigned timeout_us, void *stream)
{
    if (timeout_us < 1 || timeout_us > 1000000u) return XFA_ERR_INVALID_ARG;
    int *sp = nullptr;
    int rc = status_ptr(&sp);
    if (rc != XFA_OK) return rc;
    return cuda_code(launch_selftest_timeout(timeout_us, sp, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
