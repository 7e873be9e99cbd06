"""Edge cases of the CUDA path against the CPU oracle (GB300 only): score shapes that
drive the online softmax's running maximum, near-parallel keys (dQ as a near
cancellation), the largest problem the boundary accepts, and the rejection of the
first shape past it.  Every call goes through
the C ABI (ctypes binding)."""
import ctypes
import math

import numpy as np
import pytest
import torch

from bwd_xfa_fwd_gb300 import inputs
from tests.gpu_helpers import TOL, compare, oracle_result, run_gpu, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bwd_xfa_fwd_gb300 import binding, build
    build.build()
    binding.load()
    assert torch.cuda.is_available()


# "rising": the row maximum climbs along the row; over 128 keys it moves by up to
# scale * 256 * pi * 128 / S (in natural units; 13 in log2 units at hd = 128 and S = 1000),
# past the forward's rescale threshold of 8 on a few hundred key-tile steps of these rows.
# "falling": it never moves after the first key.  "flat": uniform rows.
@pytest.mark.parametrize("pattern", inputs.PATTERNS)
@pytest.mark.parametrize("dtype,hd,impl", [("bf16", 128, 2), ("bf16", 64, 2), ("bf16", 128, 3), ("bf16", 64, 1),
                                           ("f32", 64, 1), ("f32", 128, 1), ("f32", 64, 2), ("f32", 32, 2)])
def test_running_max_patterns(pattern, dtype, hd, impl):
    bh, S = 2, 1000
    scale = 1.0 / math.sqrt(hd)
    x = inputs.patterned((bh, S, hd), dtype, pattern, seed=77 + hd)
    got = run_gpu(x, dtype, scale, impl=impl)
    ref = oracle_result(("pattern", pattern, hd, dtype), x, scale)
    compare(got, ref, dtype)


# Near-parallel keys: the "rising" pattern with no spread in the other coordinates of K,
# so every key of a row's softmax window lies in one plane at nearly the same angle.  Then
# dQ_i = sum_j dS_ij K_j = sum_j dS_ij (K_j - K_i) (rows of dS sum to zero) is a near
# cancellation, and rounding dS to bf16 -- the operand of the dQ contraction in every bf16
# tensor-core backward -- costs up to sum_j |dS_ij| |K_jd| 2^-8 per element (bf16 keeps 8
# significant bits), 7-8 % of max|dQ| on these inputs (4-7 % measured by rounding the
# oracle's own dS).  The test asserts every other output at the usual tolerance and dQ
# element by element within that rounding bound on top of it.
@pytest.mark.parametrize("hd,impl", [(128, 2), (64, 2), (128, 3), (64, 3)])
def test_near_parallel_keys(hd, impl):
    bh, S = 2, 1000
    scale = 1.0 / math.sqrt(hd)
    x = inputs.patterned((bh, S, hd), "bf16", "rising", seed=77 + hd, k_noise=0.0)
    got = run_gpu(x, "bf16", scale, impl=impl)
    ref = oracle_result(("parallel", hd), x, scale)
    compare(got, ref, "bf16", names=("out", "lse", "dk", "dv"))
    tol = TOL["bf16"]["rel"]
    mask = np.tril(np.ones((S, S), dtype=bool))
    for b in range(bh):
        q, k, v, do = (x[n].exact[b] for n in ("q", "k", "v", "dout"))
        s = np.where(mask, scale * (q @ k.T), 0.0)
        p = np.where(mask, np.exp(s - ref["lse"][b][:, None]), 0.0)
        ds = scale * p * (do @ v.T - np.sum(do * ref["out"][b], axis=1)[:, None])
        rounding = 2.0 ** -8 * (np.abs(ds) @ np.abs(k))
        err = np.abs(got["dq"][b] - ref["dq"][b])
        bound = tol * np.max(np.abs(ref["dq"][b])) + rounding
        assert np.all(err <= bound), f"head {b}: dQ error exceeds the bf16 rounding bound by {np.max(err - bound):.3e}"


# The boundary accepts bh * S * hd < 2^31 elements.  At the largest such bh (S = 1024,
# hd = 128) every bf16 tensor spans 4.3 GB and the fp32 dQ accumulator 8.6 GB, so any
# 32-bit byte offset would wrap.  Three heads (first, middle, last, the last at the
# highest addresses) hold seeded oracle inputs; the rest are filler from the device RNG.
S_MAX, HD_MAX = 1024, 128
BH_MAX = (2 ** 31 - 1) // (S_MAX * HD_MAX)


def test_largest_accepted_problem():
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd = BH_MAX, S_MAX, HD_MAX
    assert bh * S * hd < 2 ** 31 <= (bh + 1) * S * hd
    scale = 1.0 / math.sqrt(hd)
    heads = (0, bh // 2, bh - 1)
    x = inputs.draw((len(heads), S, hd), "bf16", seed=4242)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    dev = {}
    for n in ("q", "k", "v", "dout"):
        t = torch.empty((bh, S, hd), device="cuda", dtype=torch.bfloat16)
        for h0 in range(0, bh, 2048):
            h1 = min(bh, h0 + 2048)
            t[h0:h1] = torch.randn((h1 - h0, S, hd), device="cuda", generator=gen).to(torch.bfloat16)
        t[list(heads)] = to_device(x[n], "bf16")
        dev[n] = t
    out, lse = binding.fwd(dev["q"], dev["k"], dev["v"], scale)
    dq, dk, dv = binding.bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, scale)
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    for name, t in (("out", out), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(t).all()), f"{name}: non-finite values"
    got = {n: to_f64(t[list(heads)]) for n, t in (("out", out), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    ref = oracle_result(("largest", bh), x, scale)
    compare(got, ref, "bf16")
    # on every head: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 (rows of P sum to 1, rows
    # of dS sum to 0), in fp64 on the device, a block of heads at a time
    tol = TOL["bf16"]["rel"]
    for h0 in range(0, bh, 1024):
        h1 = min(bh, h0 + 1024)
        dvb, dkb = dv[h0:h1].double(), dk[h0:h1].double()
        sv = (dvb.sum(1) - dev["dout"][h0:h1].double().sum(1)).abs().amax()
        sk = dkb.sum(1).abs().amax()
        assert float(sv) <= tol * float(dvb.abs().sum(1).amax()), f"heads {h0}..{h1}: sum dV != sum dO"
        assert float(sk) <= tol * float(dkb.abs().sum(1).amax()), f"heads {h0}..{h1}: sum dK != 0"
        del dvb, dkb


def test_first_shape_past_the_cap_is_rejected():
    from bwd_xfa_fwd_gb300 import binding
    lib = binding.load()
    buf = torch.zeros(1024, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(1024, device="cuda", dtype=torch.float32)
    p = ctypes.c_void_p(buf.data_ptr())
    pl = ctypes.c_void_p(lse.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    bh, S, hd = BH_MAX + 1, S_MAX, HD_MAX
    assert bh * S * hd >= 2 ** 31
    rc = lib.xfa_fwd(p, p, p, p, pl, bh, S, hd, ctypes.c_float(0.088), binding.XFA_BF16, st)
    assert rc == binding.XFA_ERR_INVALID_ARG
    assert lib.xfa_bwd_workspace_bytes(bh, S, hd, binding.XFA_BF16) == 0
    torch.cuda.synchronize()
    assert float(buf.float().abs().sum()) == 0.0   # nothing was written
