"""Dropout on the attention probabilities (xfa_fwd_dropout / xfa_bwd_dropout) against
the CPU oracle (GB300 only).  The mask itself is checked bit for bit: with S = hd and
V = I the forward's output is P o C, with dO = I the backward's dV is (P o C)^T, so an
element is nonzero exactly when the oracle's keep() keeps it.  Every call goes through
the C ABI (ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
from bwd_xfa_fwd_gb300 import inputs
from tests.gpu_helpers import compare, oracle_result, run_gpu, to_device, to_f64

pytestmark = pytest.mark.gpu

FAMILIES = [("bf16", 128, 2), ("bf16", 64, 2), ("bf16", 64, 1), ("f32", 32, 1), ("f32", 64, 1), ("f32", 128, 1),
            ("f32", 32, 2), ("f32", 64, 2)]


@pytest.fixture(scope="module", autouse=True)
def built():
    from bwd_xfa_fwd_gb300 import binding, build
    build.build()
    binding.load()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("S", [300, 777])
@pytest.mark.parametrize("dtype,hd,impl", FAMILIES)
def test_dropout_against_oracle(dtype, hd, impl, S, p):
    bh = 2
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), dtype, seed=500 + S + hd)
    seed = 0x5EED0000 + S
    got = run_gpu(x, dtype, scale, impl=impl, dropout=(p, seed))
    ref = oracle_result(("drop", S, hd, dtype), x, scale, dropout=(p, seed))
    compare(got, ref, dtype)


def _kept_reference(bh, S, p, seed):
    """keep(seed, (b*S + i)*S + j, p) of the pinned oracle, for j <= i (above the
    diagonal the probabilities are 0 whatever the mask)."""
    k = np.zeros((bh, S, S), dtype=bool)
    for b in range(bh):
        for i in range(S):
            base = (b * S + i) * S
            for j in range(i + 1):
                k[b, i, j] = oracle.keep(seed, base + j, p)
    return k


@pytest.mark.parametrize("dtype,hd,impl", FAMILIES)
def test_dropout_mask_bit_for_bit(dtype, hd, impl):
    from bwd_xfa_fwd_gb300 import binding
    bh, S, p, seed = 2, hd, 0.3, 0xA5A5A5A5DEADBEEF
    x = inputs.draw((bh, S, hd), dtype, seed=7, stds=(0.3, 0.3, 1.0, 1.0))
    eye = np.broadcast_to(np.eye(S, dtype=np.float32), (bh, S, S)).copy()
    ident = inputs._stored(eye, dtype)
    q, k = to_device(x["q"], dtype), to_device(x["k"], dtype)
    v = to_device(ident, dtype)
    do = to_device(ident, dtype)
    scale = 1.0 / math.sqrt(hd)
    out, lse = binding.fwd(q, k, v, scale, impl, dropout_p=p, seed=seed)
    dq, dk, dv = binding.bwd(q, k, v, out, do, lse, scale, impl, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    want = _kept_reference(bh, S, p, seed)
    lower = np.tril(np.ones((S, S), dtype=bool))
    got_fwd = to_f64(out) != 0.0                      # O = P o C   (V = I)
    got_bwd = np.swapaxes(to_f64(dv), 1, 2) != 0.0    # dV^T = P o C   (dO = I)
    for name, got in (("forward", got_fwd), ("backward", got_bwd)):
        bad = (got != want) & lower
        assert not bad.any(), f"{name}: {int(bad.sum())} mask bits differ, first at {np.argwhere(bad)[0].tolist()}"
    kept = want[:, lower].mean()
    assert abs(kept - (1 - p)) < 0.05, kept


@pytest.mark.parametrize("dtype,hd,impl", [("bf16", 128, 2), ("f32", 64, 1)])
def test_rate_zero_is_the_plain_operator(dtype, hd, impl):
    from bwd_xfa_fwd_gb300 import binding
    x = inputs.draw((2, 200, hd), dtype, seed=11)
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    lib = binding.load()
    outs = []
    for use_dropout_entry in (False, True):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:-1], device="cuda", dtype=torch.float32)
        st = binding._stream(q)
        args = (binding._p(q), binding._p(k), binding._p(v), binding._p(out), binding._p(lse), 2, 200, hd, 0.1,
                binding._DTYPE[q.dtype])
        if use_dropout_entry:
            rc = lib.xfa_fwd_dropout(*args, 0.0, 99, impl, st)
        else:
            rc = lib.xfa_fwd_impl(*args, impl, st)
        assert rc == binding.XFA_OK
        grads = binding.bwd(q, k, v, out, do, lse, 0.1, impl, dropout_p=0.0, seed=99)
        torch.cuda.synchronize()
        outs.append([out, lse, *grads])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_same_seed_same_result_other_seed_other_mask():
    x = inputs.draw((1, 256, 64), "bf16", seed=12)
    a = run_gpu(x, "bf16", 0.125, dropout=(0.2, 1))
    b = run_gpu(x, "bf16", 0.125, dropout=(0.2, 1))
    c = run_gpu(x, "bf16", 0.125, dropout=(0.2, 2))
    for n in a:
        assert np.array_equal(a[n], b[n]), n
    assert not np.array_equal(a["out"], c["out"])
    assert np.array_equal(a["lse"], c["lse"])   # the softmax itself is not dropped


def test_full_size_sampled_heads_with_dropout():
    """The S = 8192 workload with p = 0.1: four heads (first, last and two between) against
    the oracle, whose per-element draws make a head several times dearer than without."""
    w = inputs.WORKLOADS[5]
    x = inputs.workload_inputs(w)
    got = run_gpu(x, w.dtype, w.scale, dropout=(0.1, 2024))
    heads = [0, 11, 22, 31]
    ref = oracle_result(("w5drop",), x, w.scale, heads=heads, dropout=(0.1, 2024))
    compare(got, ref, w.dtype, heads=heads)


def test_dropout_rejections():
    from bwd_xfa_fwd_gb300 import binding
    x = inputs.draw((1, 128, 64), "bf16", seed=3)
    q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
    for bad in (1.0, -0.1, float("nan"), 1.5):
        with pytest.raises(binding.XfaError) as e:
            binding.fwd(q, k, v, 0.1, dropout_p=bad, seed=1)
        assert e.value.code == binding.XFA_ERR_INVALID_ARG
    out, lse = binding.fwd(q, k, v, 0.1, dropout_p=0.2, seed=1)
    with pytest.raises(binding.XfaError) as e:
        binding.bwd(q, k, v, out, do, lse, 0.1, binding.IMPL_TCGEN05_DET, dropout_p=0.2, seed=1)
    assert e.value.code == binding.XFA_ERR_UNSUPPORTED


def test_tape_node_with_dropout():
    from bwd_xfa_fwd_gb300 import binding, tape
    x = inputs.draw((2, 300, 128), "bf16", seed=21)
    dev = {n: to_device(x[n], "bf16") for n in ("q", "k", "v", "dout")}
    qv, kv, vv = (tape.Var(dev[n]) for n in ("q", "k", "v"))
    o = tape.flash_attention(qv, kv, vv, dropout_p=0.25, seed=77)
    o.backward(seed=dev["dout"])
    torch.cuda.synchronize()
    ref = run_gpu(x, "bf16", binding.default_scale(128), dropout=(0.25, 77))
    assert np.array_equal(to_f64(o.value), ref["out"])
    for var, n in ((qv, "dq"), (kv, "dk"), (vv, "dv")):
        assert np.array_equal(to_f64(var.grad), ref[n]), n


def _keep_pair(x, dtype, hd, p, seed, impl=2, fill=False):
    """Forward + backward with the keep-bit cache -- stored by the forward, or (fill) drawn by
    xfa_dropout_keep_fill and read by both -- and the re-drawing pair on the same inputs."""
    from bwd_xfa_fwd_gb300 import binding
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    bh, S, _ = q.shape
    scale = 1.0 / math.sqrt(hd)
    keep = torch.full((binding.dropout_keep_bytes(bh, S),), 0xAB, device="cuda", dtype=torch.uint8)
    if fill:
        binding.dropout_keep_fill(bh, S, p, seed, keep)
    out_k, lse_k = binding.fwd(q, k, v, scale, impl, dropout_p=p, seed=0 if fill else seed, keep_bits=keep,
                               keep_cached=fill)
    g_k = binding.bwd(q, k, v, out_k, do, lse_k, scale, impl, dropout_p=p, keep_bits=keep)
    out_d, lse_d = binding.fwd(q, k, v, scale, impl, dropout_p=p, seed=seed)
    g_d = binding.bwd(q, k, v, out_d, do, lse_d, scale, impl, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    return keep, (out_k, lse_k) + tuple(g_k), (out_d, lse_d) + tuple(g_d)


def _assert_same_as_redrawn(cached, redrawn):
    """Forward, dK and dV bit for bit; dQ is summed with reduce-adds in a data-dependent
    order, so two runs of the same backward differ by bf16 rounding steps."""
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), cached, redrawn):
        if name == "dq":
            tol = 1e-2 * float(b.float().abs().max())
            assert torch.allclose(a.float(), b.float(), rtol=0, atol=tol), name
        else:
            assert torch.equal(a, b), name


@pytest.mark.parametrize("fill", [False, True])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("S", [1, 127, 300, 777, 1024])
def test_cached_keep_bits_give_the_redrawn_results(hd, S, fill):
    x = inputs.draw((2, S, hd), "bf16", seed=900 + S + hd)
    _, cached, redrawn = _keep_pair(x, "bf16", hd, 0.2, 0xC0FFEE + S, fill=fill)
    _assert_same_as_redrawn(cached, redrawn)


@pytest.mark.parametrize("S", [1, 200, 300, 777])
def test_fill_writes_what_the_forward_stores(S):
    """xfa_dropout_keep_fill and the storing forward write the same bits into every word at or
    below the diagonal (w >= 4 kt) and leave the others alone."""
    from bwd_xfa_fwd_gb300 import binding
    bh, hd, p, seed = 3, 64, 0.25, 0xBADC0DE + S
    x = inputs.draw((bh, S, hd), "bf16", seed=S)
    q, k, v = (to_device(x[n], "bf16") for n in ("q", "k", "v"))
    n = binding.dropout_keep_bytes(bh, S)
    a = torch.full((n,), 0x5A, device="cuda", dtype=torch.uint8)
    b = torch.full((n,), 0x5A, device="cuda", dtype=torch.uint8)
    binding.dropout_keep_fill(bh, S, p, seed, a)
    binding.fwd(q, k, v, 0.125, dropout_p=p, seed=seed, keep_bits=b)
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    nkt = (S + 127) // 128
    nw = 4 * nkt
    wa = a.view(torch.int32).reshape(bh, nkt, nw, 128)
    wb = b.view(torch.int32).reshape(bh, nkt, nw, 128)
    assert torch.equal(wa, wb)
    untouched = torch.full((), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    for kt in range(nkt):
        assert bool((wa[:, kt, : 4 * kt] == untouched).all()), kt          # above the diagonal: not written
        assert not bool((wa[:, kt, 4 * kt:] == untouched).all()), kt      # at or below: written


def test_cached_keep_bits_are_the_oracle_mask():
    """Decode the forward's keep-bit cache (bit i of word ((b*nkt + kt)*nw + w)*128 + c is
    the decision of (b, row 32w + i, key 128kt + c), nkt = ceil(S/128), nw = 4 nkt) and compare
    every decision at or below the diagonal with the oracle's keep()."""
    bh, S, hd, p, seed = 2, 300, 64, 0.3, 0x1234ABCD5678
    x = inputs.draw((bh, S, hd), "bf16", seed=31)
    keep, _, _ = _keep_pair(x, "bf16", hd, p, seed)
    nkt = (S + 127) // 128
    nw = 4 * nkt
    words = keep.view(torch.int32).cpu().numpy().view(np.uint32).reshape(bh, nkt, nw, 128)
    rows = np.arange(S)
    bits = (words[:, :, rows // 32, :] >> (rows % 32)[None, None, :, None].astype(np.uint32)) & 1   # [b, kt, row, c]
    got = bits.transpose(0, 2, 1, 3).reshape(bh, S, nkt * 128)[:, :, :S].astype(bool)
    want = _kept_reference(bh, S, p, seed)
    lower = np.tril(np.ones((S, S), dtype=bool))
    bad = (got != want) & lower
    assert not bad.any(), f"{int(bad.sum())} cached bits differ, first at {np.argwhere(bad)[0].tolist()}"


@pytest.mark.parametrize("fill", [False, True])
def test_cached_keep_bits_full_size(fill):
    """The S = 8192 workload with p = 0.1: the pair from the cache is the re-drawing one."""
    w = inputs.WORKLOADS[5]
    x = inputs.workload_inputs(w)
    _, cached, redrawn = _keep_pair(x, w.dtype, w.hd, 0.1, 2024, fill=fill)
    _assert_same_as_redrawn(cached, redrawn)


def test_cached_keep_bits_rejections():
    from bwd_xfa_fwd_gb300 import binding
    x = inputs.draw((1, 256, 64), "bf16", seed=5)
    q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
    need = binding.dropout_keep_bytes(1, 256)
    keep = torch.zeros(need, device="cuda", dtype=torch.uint8)
    with pytest.raises(binding.XfaError) as e:
        binding.fwd(q, k, v, 0.1, dropout_p=0.2, seed=1, keep_bits=keep[: need - 16])
    assert e.value.code == binding.XFA_ERR_INVALID_ARG
    with pytest.raises(binding.XfaError) as e:
        binding.fwd(q, k, v, 0.1, dropout_p=0.2, seed=1, keep_bits=torch.zeros(need + 4, device="cuda",
                                                                                 dtype=torch.uint8)[4:])
    assert e.value.code == binding.XFA_ERR_INVALID_ARG
    for cached in (False, True):
        with pytest.raises(binding.XfaError) as e:
            binding.fwd(q, k, v, 0.1, binding.IMPL_SIMT, dropout_p=0.2, seed=1, keep_bits=keep, keep_cached=cached)
        assert e.value.code == binding.XFA_ERR_UNSUPPORTED
    with pytest.raises(binding.XfaError) as e:
        binding.dropout_keep_fill(1, 256, 0.2, 1, keep[: need - 16])
    assert e.value.code == binding.XFA_ERR_INVALID_ARG
    out, lse = binding.fwd(q, k, v, 0.1, dropout_p=0.2, seed=1, keep_bits=keep)
    for impl in (binding.IMPL_SIMT, binding.IMPL_TCGEN05_DET):
        with pytest.raises(binding.XfaError) as e:
            binding.bwd(q, k, v, out, do, lse, 0.1, impl, dropout_p=0.2, keep_bits=keep)
        assert e.value.code == binding.XFA_ERR_UNSUPPORTED
    x32 = inputs.draw((1, 256, 64), "f32", seed=5)
    q32, k32, v32 = (to_device(x32[n], "f32") for n in ("q", "k", "v"))
    with pytest.raises(binding.XfaError) as e:
        binding.fwd(q32, k32, v32, 0.1, dropout_p=0.2, seed=1, keep_bits=keep)
    assert e.value.code == binding.XFA_ERR_UNSUPPORTED


def test_tape_node_with_a_kept_mask():
    """The tape node with keep_mask: the forward stores its mask, the backward reads it; the
    results are the re-drawing node's (dQ up to the order of its reduce-adds)."""
    from bwd_xfa_fwd_gb300 import binding, tape
    x = inputs.draw((2, 300, 128), "bf16", seed=22)
    dev = {n: to_device(x[n], "bf16") for n in ("q", "k", "v", "dout")}
    res = []
    for keep_mask in (False, True):
        qv, kv, vv = (tape.Var(dev[n].clone()) for n in ("q", "k", "v"))
        o = tape.flash_attention(qv, kv, vv, dropout_p=0.25, seed=78, keep_mask=keep_mask)
        assert ("keep_bits" in o.saved) == keep_mask
        o.backward(seed=dev["dout"])
        torch.cuda.synchronize()
        assert binding.status() == binding.XFA_OK
        res.append((o.value, o.saved["lse"], qv.grad, kv.grad, vv.grad))
    _assert_same_as_redrawn(res[1], res[0])
