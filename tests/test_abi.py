"""The C ABI library: it builds, loads, exports every declared entry point, and
rejects bad arguments on the host (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

from bwd_xfa_fwd_gb300 import build as xbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bwd_xfa_fwd_gb300 import binding
    xbuild.build()
    return binding.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "xfa.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(xfa_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror(lib):
    from bwd_xfa_fwd_gb300 import binding
    assert lib.xfa_version() == 100
    assert "timeout" in binding.strerror(binding.XFA_ERR_TIMEOUT)
    assert binding.strerror(1000 + 2)  # a CUDA error string


def test_workspace_bytes(lib):
    from bwd_xfa_fwd_gb300 import binding
    ws = lib.xfa_bwd_workspace_bytes
    # D and Lg: bh * roundup(S, 128) fp32 each (256-aligned); bf16 adds the fp32 dQ accumulator
    assert ws(2, 64, 32, binding.XFA_F32) == 2 * 128 * 4 * 2
    assert ws(32, 8192, 128, binding.XFA_BF16) == 2 * 32 * 8192 * 4 + 32 * 8192 * 128 * 4
    assert ws(0, 64, 32, 0) == 0 and ws(1, 64, 48, 0) == 0


def _fwd(lib, ptrs, bh=1, S=8, hd=64, scale=0.125, dtype=1, impl=0):
    return lib.xfa_fwd_impl(*ptrs, bh, S, hd, ctypes.c_float(scale), dtype, impl, None)


def test_host_validation(lib):
    from bwd_xfa_fwd_gb300 import binding as b
    good = [ctypes.c_void_p(4096 * (i + 1)) for i in range(5)]
    assert _fwd(lib, good, hd=48) == b.XFA_ERR_UNSUPPORTED
    assert _fwd(lib, good, bh=0) == b.XFA_ERR_INVALID_ARG
    assert _fwd(lib, good, S=0) == b.XFA_ERR_INVALID_ARG
    assert _fwd(lib, good, scale=0.0) == b.XFA_ERR_INVALID_ARG
    assert _fwd(lib, good, scale=float("nan")) == b.XFA_ERR_INVALID_ARG
    assert _fwd(lib, good, dtype=7) == b.XFA_ERR_INVALID_ARG
    assert _fwd(lib, good, bh=1 << 12, S=1 << 12, hd=128) == b.XFA_ERR_INVALID_ARG   # 2^31 elements
    bad = list(good)
    bad[2] = ctypes.c_void_p(4096 + 8)      # misaligned
    assert _fwd(lib, bad) == b.XFA_ERR_INVALID_ARG
    bad[2] = ctypes.c_void_p(0)             # null
    assert _fwd(lib, bad) == b.XFA_ERR_INVALID_ARG
    p = [ctypes.c_void_p(4096 * (i + 1)) for i in range(9)]
    rc = lib.xfa_bwd_impl(*p, 1, 8, 64, ctypes.c_float(0.125), 1, ctypes.c_void_p(0), 0, 0, None)
    assert rc == b.XFA_ERR_WORKSPACE
    assert lib.xfa_accumulate(None, None, 4, 0, None) == b.XFA_ERR_INVALID_ARG
    assert lib.xfa_accumulate(None, None, 0, 0, None) == b.XFA_OK
    assert lib.xfa_selftest_timeout(0, None) == b.XFA_ERR_INVALID_ARG


def test_dropout_keep_bytes_and_validation(lib):
    """The keep-bit cache of the dropout pair: its size (key tiles of 128 x query-row words of
    32, 128 words each) and the host checks of the buffer and of the family."""
    from bwd_xfa_fwd_gb300 import binding as b
    kb = lib.xfa_dropout_keep_bytes
    assert kb(2, 300) == 2 * 3 * 12 * 128 * 4      # ceil(300/128) key tiles, 4 words of 32 rows each
    assert kb(32, 8192) == 32 * 64 * 256 * 128 * 4
    assert kb(0, 64) == 0 and kb(1, 0) == 0 and kb(1 << 13, 1 << 13) == 0
    good = [ctypes.c_void_p(4096 * (i + 1)) for i in range(5)]
    need = kb(1, 8)
    keep = ctypes.c_void_p(1 << 20)

    def fwd_keep(buf, nbytes, impl=b.IMPL_SIMT, p=0.1):
        return lib.xfa_fwd_dropout_keep(*good, 1, 8, 64, ctypes.c_float(0.125), b.XFA_BF16, ctypes.c_float(p), 7,
                                        buf, nbytes, impl, None)

    assert fwd_keep(None, need) == b.XFA_ERR_INVALID_ARG
    assert fwd_keep(ctypes.c_void_p((1 << 20) + 4), need) == b.XFA_ERR_INVALID_ARG
    assert fwd_keep(keep, need - 1) == b.XFA_ERR_INVALID_ARG
    assert fwd_keep(keep, need, p=1.0) == b.XFA_ERR_INVALID_ARG
    assert fwd_keep(keep, need) == b.XFA_ERR_UNSUPPORTED            # the SIMT family keeps no bits
    p9 = [ctypes.c_void_p(4096 * (i + 1)) for i in range(9)]
    ws = lib.xfa_bwd_workspace_bytes(1, 8, 64, b.XFA_BF16)

    def bwd_keep(buf, nbytes, impl=b.IMPL_SIMT):
        return lib.xfa_bwd_dropout_cached(*p9, 1, 8, 64, ctypes.c_float(0.125), b.XFA_BF16, ctypes.c_float(0.1),
                                        buf, nbytes, ctypes.c_void_p(1 << 24), ws, impl, None)

    assert lib.xfa_dropout_keep_fill(1, 8, ctypes.c_float(0.1), 7, None, need, None) == b.XFA_ERR_INVALID_ARG
    assert lib.xfa_dropout_keep_fill(1, 8, ctypes.c_float(0.1), 7, keep, need - 4, None) == b.XFA_ERR_INVALID_ARG
    assert lib.xfa_dropout_keep_fill(1, 8, ctypes.c_float(0.0), 7, keep, need, None) == b.XFA_OK   # nothing to draw
    assert bwd_keep(None, need) == b.XFA_ERR_INVALID_ARG
    assert bwd_keep(keep, need - 16) == b.XFA_ERR_INVALID_ARG
