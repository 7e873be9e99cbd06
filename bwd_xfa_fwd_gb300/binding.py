"""ctypes binding of ``libxfa.so`` (C ABI in ``include/xfa.h``).

Argument marshalling only: torch supplies device memory and the current CUDA
stream; every step of attention runs in the library's kernels.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libxfa.so")

XFA_F32, XFA_BF16 = 0, 1
IMPL_AUTO, IMPL_SIMT, IMPL_TCGEN05, IMPL_TCGEN05_DET = 0, 1, 2, 3
XFA_OK, XFA_ERR_INVALID_ARG, XFA_ERR_UNSUPPORTED, XFA_ERR_TIMEOUT, XFA_ERR_WORKSPACE, XFA_ERR_DEVICE = range(6)
XFA_ERR_CUDA_BASE = 1000

_DTYPE = {torch.float32: XFA_F32, torch.bfloat16: XFA_BF16}
_lib = None


class XfaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with bwd_xfa_fwd_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i, f, sz, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
    sigs = {
        "xfa_fwd": ([vp, vp, vp, vp, vp, i, i, i, f, i, vp], i),
        "xfa_fwd_impl": ([vp, vp, vp, vp, vp, i, i, i, f, i, i, vp], i),
        "xfa_fwd_dropout": ([vp, vp, vp, vp, vp, i, i, i, f, i, f, u64, i, vp], i),
        "xfa_bwd_workspace_bytes": ([i, i, i, i], sz),
        "xfa_bwd": ([vp] * 9 + [i, i, i, f, i, vp, sz, vp], i),
        "xfa_bwd_impl": ([vp] * 9 + [i, i, i, f, i, vp, sz, i, vp], i),
        "xfa_bwd_dropout": ([vp] * 9 + [i, i, i, f, i, f, u64, vp, sz, i, vp], i),
        "xfa_dropout_keep_bytes": ([i, i], sz),
        "xfa_fwd_dropout_keep": ([vp, vp, vp, vp, vp, i, i, i, f, i, f, u64, vp, sz, i, vp], i),
        "xfa_fwd_dropout_cached": ([vp, vp, vp, vp, vp, i, i, i, f, i, f, vp, sz, i, vp], i),
        "xfa_bwd_dropout_cached": ([vp] * 9 + [i, i, i, f, i, f, vp, sz, vp, sz, i, vp], i),
        "xfa_dropout_keep_fill": ([i, i, f, u64, vp, sz, vp], i),
        "xfa_bwd_prep": ([vp, vp, vp, vp, i, i, i, i, vp, sz, i, vp], i),
        "xfa_bwd_main": ([vp] * 7 + [i, i, i, f, i, vp, sz, i, vp], i),
        "xfa_bwd_finish": ([vp, i, i, i, i, vp, sz, i, vp], i),
        "xfa_rowdot": ([vp, vp, vp, i, i, i, i, vp], i),
        "xfa_accumulate": ([vp, vp, sz, i, vp], i),
        "xfa_status": ([vp], i),
        "xfa_last_status": ([vp], i),
        "xfa_selftest_timeout": ([ctypes.c_uint, vp], i),
        "xfa_strerror": ([i], ctypes.c_char_p),
        "xfa_version": ([], i),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().xfa_strerror(int(code)).decode()


def _check(code: int, what: str):
    if code != XFA_OK:
        raise XfaError(code, what)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: torch.Tensor) -> int:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("keep_bits must be a contiguous CUDA tensor")
    return t.numel() * t.element_size()


def _shape3(q: torch.Tensor):
    """[bh, S, hd] or [B, H, S, hd] (contiguous) -> (bh, S, hd)."""
    if q.dim() == 3:
        return tuple(q.shape)
    if q.dim() == 4:
        return q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
    raise ValueError("expected a [bh, S, hd] or [B, H, S, hd] tensor")


def _check_tensors(*ts):
    ref = ts[0]
    if ref.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {ref.dtype}")
    for t in ts:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != ref.dtype or t.shape != ref.shape:
            raise ValueError("tensors must be contiguous CUDA tensors of one shape and dtype")


def default_scale(hd: int) -> float:
    return 1.0 / math.sqrt(hd)


def dropout_keep_bytes(bh: int, S: int) -> int:
    """Bytes of the keep-bit cache of a dropout forward / backward pair (xfa_dropout_keep_bytes)."""
    return int(load().xfa_dropout_keep_bytes(bh, S))


def dropout_keep_fill(bh: int, S: int, dropout_p: float, seed: int, keep_bits, stream_of=None):
    """Draw every keep decision of a (bh, S) dropout into ``keep_bits`` (xfa_dropout_keep_fill),
    on the current stream of ``stream_of``'s device (default: keep_bits')."""
    ref = keep_bits if stream_of is None else stream_of
    _check(load().xfa_dropout_keep_fill(bh, S, float(dropout_p), int(seed) % 2 ** 64, _p(keep_bits),
                                        _nbytes(keep_bits), _stream(ref)), "xfa_dropout_keep_fill")


def fwd(q, k, v, scale: float | None = None, impl: int = IMPL_AUTO, out=None, lse=None, dropout_p: float = 0.0,
        seed: int = 0, keep_bits=None, keep_cached: bool = False):
    """Forward: returns (O, L).  O has q's shape/dtype; L is fp32 [..., S].  ``dropout_p`` > 0
    applies dropout of that rate to the attention probabilities (xfa_fwd_dropout); the
    backward must get the same ``dropout_p`` and ``seed``.  With ``keep_bits`` (a CUDA uint8
    tensor of at least :func:`dropout_keep_bytes` bytes) the forward also stores its keep
    decisions there (xfa_fwd_dropout_keep), or, with ``keep_cached``, reads them from it
    instead of drawing (xfa_fwd_dropout_cached; filled by :func:`dropout_keep_fill`)."""
    _check_tensors(q, k, v)
    bh, S, hd = _shape3(q)
    scale = default_scale(hd) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:-1], device=q.device, dtype=torch.float32) if lse is None else lse
    if dropout_p and keep_bits is not None and keep_cached:
        _check(load().xfa_fwd_dropout_cached(_p(q), _p(k), _p(v), _p(out), _p(lse), bh, S, hd, scale,
                                             _DTYPE[q.dtype], float(dropout_p), _p(keep_bits), _nbytes(keep_bits),
                                             impl, _stream(q)), "xfa_fwd_dropout_cached")
    elif dropout_p and keep_bits is not None:
        _check(load().xfa_fwd_dropout_keep(_p(q), _p(k), _p(v), _p(out), _p(lse), bh, S, hd, scale, _DTYPE[q.dtype],
                                           float(dropout_p), int(seed) % 2 ** 64, _p(keep_bits), _nbytes(keep_bits),
                                           impl, _stream(q)), "xfa_fwd_dropout_keep")
    elif dropout_p:
        _check(load().xfa_fwd_dropout(_p(q), _p(k), _p(v), _p(out), _p(lse), bh, S, hd, scale, _DTYPE[q.dtype],
                                      float(dropout_p), int(seed) % 2 ** 64, impl, _stream(q)), "xfa_fwd_dropout")
    else:
        _check(load().xfa_fwd_impl(_p(q), _p(k), _p(v), _p(out), _p(lse), bh, S, hd, scale, _DTYPE[q.dtype], impl,
                                   _stream(q)), "xfa_fwd")
    return out, lse


def workspace_bytes(bh: int, S: int, hd: int, dtype: torch.dtype) -> int:
    return int(load().xfa_bwd_workspace_bytes(bh, S, hd, _DTYPE[dtype]))


def bwd(q, k, v, out, dout, lse, scale: float | None = None, impl: int = IMPL_AUTO, workspace=None, grads=None,
        dropout_p: float = 0.0, seed: int = 0, keep_bits=None):
    """Backward: returns (dQ, dK, dV), each of q's shape/dtype (overwritten).  ``dropout_p`` and
    ``seed`` must be those of the forward (xfa_bwd_dropout when ``dropout_p`` > 0); with
    ``keep_bits``, the cached decisions are read instead of drawn (xfa_bwd_dropout_cached, no
    seed needed)."""
    _check_tensors(q, k, v, out, dout)
    bh, S, hd = _shape3(q)
    scale = default_scale(hd) if scale is None else float(scale)
    need = workspace_bytes(bh, S, hd, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    dq, dk, dv = grads if grads is not None else (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q))
    if dropout_p and keep_bits is not None:
        _check(load().xfa_bwd_dropout_cached(_p(q), _p(k), _p(v), _p(out), _p(dout), _p(lse), _p(dq), _p(dk),
                                             _p(dv), bh, S, hd, scale, _DTYPE[q.dtype], float(dropout_p),
                                             _p(keep_bits), _nbytes(keep_bits), _p(workspace), workspace.numel(), impl,
                                             _stream(q)), "xfa_bwd_dropout_cached")
    elif dropout_p:
        _check(load().xfa_bwd_dropout(_p(q), _p(k), _p(v), _p(out), _p(dout), _p(lse), _p(dq), _p(dk), _p(dv), bh, S,
                                      hd, scale, _DTYPE[q.dtype], float(dropout_p), int(seed) % 2 ** 64,
                                      _p(workspace), workspace.numel(), impl, _stream(q)), "xfa_bwd_dropout")
    else:
        _check(load().xfa_bwd_impl(_p(q), _p(k), _p(v), _p(out), _p(dout), _p(lse), _p(dq), _p(dk), _p(dv), bh, S,
                                   hd, scale, _DTYPE[q.dtype], _p(workspace), workspace.numel(), impl, _stream(q)),
               "xfa_bwd")
    return dq, dk, dv


def bwd_stages(q, k, v, out, dout, lse, scale, workspace, grads, impl: int = IMPL_AUTO, hook=None):
    """The backward as its three enqueued stages (prep, main, finish); ``hook(name)``
    is called before each stage and after the last with ``"end"`` (e.g. to record
    CUDA events).  Same result as :func:`bwd`."""
    _check_tensors(q, k, v, out, dout)
    bh, S, hd = _shape3(q)
    dq, dk, dv = grads
    dt = _DTYPE[q.dtype]
    lib, st, ws, nws = load(), _stream(q), _p(workspace), workspace.numel()
    hook = hook or (lambda name: None)
    hook("prep")
    _check(lib.xfa_bwd_prep(_p(out), _p(dout), _p(lse), _p(dq), bh, S, hd, dt, ws, nws, impl, st), "xfa_bwd_prep")
    hook("main")
    _check(lib.xfa_bwd_main(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), bh, S, hd, float(scale), dt, ws,
                            nws, impl, st), "xfa_bwd_main")
    hook("finish")
    _check(lib.xfa_bwd_finish(_p(dq), bh, S, hd, dt, ws, nws, impl, st), "xfa_bwd_finish")
    hook("end")
    return dq, dk, dv


def rowdot(out, dout):
    """D = sum_d dout * out per row, fp32 [..., S]."""
    _check_tensors(out, dout)
    bh, S, hd = _shape3(out)
    d = torch.empty(out.shape[:-1], device=out.device, dtype=torch.float32)
    _check(load().xfa_rowdot(_p(out), _p(dout), _p(d), bh, S, hd, _DTYPE[out.dtype], _stream(out)), "xfa_rowdot")
    return d


def accumulate_(dst, src):
    """dst += src on the device (fan-out gradient sum)."""
    _check_tensors(dst, src)
    _check(load().xfa_accumulate(_p(dst), _p(src), dst.numel(), _DTYPE[dst.dtype], _stream(dst)),
           "xfa_accumulate")
    return dst


def status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status word."""
    s = torch.cuda.current_stream(device)
    return int(load().xfa_last_status(ctypes.c_void_p(s.cuda_stream)))


def selftest_timeout(timeout_us: int, device=None) -> int:
    s = torch.cuda.current_stream(device)
    return int(load().xfa_selftest_timeout(int(timeout_us), ctypes.c_void_p(s.cuda_stream)))
