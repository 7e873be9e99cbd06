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
