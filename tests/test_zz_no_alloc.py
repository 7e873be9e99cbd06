"""xfa_bwd_noalloc: the backward for callers that cannot allocate device memory
(a framework that reserved the device memory for its own allocator, a plug-in
host that forbids allocation in its callbacks, code that cannot take the
implicit synchronisation of cudaMalloc).  Its scratch is a fixed device array
inside the library instead of a caller-provided workspace.

Checked through the C ABI against xfa_bwd on the same inputs, on two calls in
a row (the array keeps the previous call's contents, so the second call shows
that everything read is rewritten or cleared first), and the second call is
checked to leave the device's free memory and torch's allocator unchanged.
This file is collected last so that a run stopping at the first failure has
run every other test."""
import ctypes
import math

import pytest
import torch

from bwd_xfa_fwd_gb300 import inputs
from tests.gpu_helpers import compare, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from bwd_xfa_fwd_gb300 import binding, build
    build.build()
    lib = binding.load()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.xfa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, f, i, vp]
    lib.xfa_bwd_noalloc.restype = i
    return lib


def _call(lib, t, grads, bh, S, hd, scale, dtype_code):
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.xfa_bwd_noalloc(p(t["q"]), p(t["k"]), p(t["v"]), p(t["out"]), p(t["dout"]), p(t["lse"]),
                               p(grads[0]), p(grads[1]), p(grads[2]), bh, S, hd, scale, dtype_code, stream)


@pytest.mark.parametrize("dtype,hd,S,bh", [("bf16", 128, 1000, 4), ("bf16", 64, 777, 3), ("f32", 64, 300, 2)])
def test_noalloc_matches_bwd_twice(lib, dtype, hd, S, bh):
    from bwd_xfa_fwd_gb300 import binding
    scale = 1.0 / math.sqrt(hd)
    code = binding.XFA_BF16 if dtype == "bf16" else binding.XFA_F32
    t = {}
    for call in range(2):
        x = inputs.draw((bh, S, hd), dtype, seed=500 + call + hd)   # different inputs per call
        t = {n: to_device(x[n], dtype) for n in ("q", "k", "v", "dout")}
        t["out"], t["lse"] = binding.fwd(t["q"], t["k"], t["v"], scale)
        want = binding.bwd(t["q"], t["k"], t["v"], t["out"], t["dout"], t["lse"], scale)
        got = tuple(torch.full_like(t["q"], float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free0, held0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert _call(lib, t, got, bh, S, hd, scale, code) == binding.XFA_OK
        torch.cuda.synchronize()
        if call == 1:
            # the first call on a device may load the library module that holds the array;
            # a later call must leave the device's free memory and torch's allocator as they were
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_allocated() == held0
        assert binding.status() == binding.XFA_OK
        compare({n: to_f64(g) for n, g in zip(("dq", "dk", "dv"), got)},
                {n: to_f64(w) for n, w in zip(("dq", "dk", "dv"), want)}, dtype, names=("dq", "dk", "dv"))


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    from bwd_xfa_fwd_gb300 import binding
    big = binding.workspace_bytes(32, 8192, 128, torch.bfloat16)
    assert big > 32 * 1024 * 1024
    q = torch.zeros(16, device="cuda")   # never touched: the size check comes first
    t = {n: q for n in ("q", "k", "v", "out", "dout", "lse")}
    rc = _call(lib, t, (q, q, q), 32, 8192, 128, 0.088, binding.XFA_BF16)
    assert rc == binding.XFA_ERR_WORKSPACE
    rc = _call(lib, t, (q, q, q), 1, 64, 48, 0.1, binding.XFA_BF16)
    assert rc == binding.XFA_ERR_UNSUPPORTED
