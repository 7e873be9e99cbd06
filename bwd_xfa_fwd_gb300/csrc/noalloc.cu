// xfa_bwd_noalloc: the backward with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they need the
// backward: a host framework that has already reserved the device memory for
// its own allocator, a plug-in whose host forbids device allocation inside
// its callbacks, or latency-critical code that cannot afford cudaMalloc's
// implicit device-wide synchronisation.  This entry point needs no workspace
// from them: the D / L*log2(e) rows and the fp32 dQ accumulator live in one
// file-scope device array of XFA_NOALLOC_SCRATCH_BYTES, kept on a device until
// the process exits.
//
// The array's host-side name is only a stand-in for the symbol; its device
// address is resolved with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and passed to the kernels.  With
// lazy module loading (CUDA's default) that first resolution is also what
// loads this file's module, and so reserves the array on the device: the
// first call on a device may allocate and synchronise, and fails with
// cudaErrorMemoryAllocation when the device is full.  Later calls allocate
// nothing.  All calls share the array and it keeps the last call's contents;
// the pre-pass of every call rewrites D and L and clears the dQ accumulator
// before use.
// Calls that overlap on the GPU (other streams, other host threads) race on
// the array.
#include <mutex>

#include <cuda_runtime.h>

#include "xfa.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[XFA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device.
int scratch_ptr(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
    if (dev < 0 || dev >= kMaxDevices) return XFA_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return XFA_ERR_CUDA_BASE + (int)e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return XFA_OK;
}

}  // namespace

extern "C" int xfa_bwd_noalloc(const void *q, const void *k, const void *v, const void *out, const void *dout,
                               const float *lse, void *dq, void *dk, void *dv, int bh, int S, int hd, float scale,
                               int dtype, void *stream)
{
    const size_t need = xfa_bwd_workspace_bytes(bh, S, hd, dtype);
    if (need == 0) {
        // invalid shape: let the regular entry point name the error (it checks before touching memory)
        return xfa_bwd(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, nullptr, 0, stream);
    }
    if (need > (size_t)XFA_NOALLOC_SCRATCH_BYTES) return XFA_ERR_WORKSPACE;
    void *ws = nullptr;
    int rc = scratch_ptr(&ws);
    if (rc != XFA_OK) return rc;
    return xfa_bwd(q, k, v, out, dout, lse, dq, dk, dv, bh, S, hd, scale, dtype, ws,
                   (size_t)XFA_NOALLOC_SCRATCH_BYTES, stream);
}
