"""A whole forward + backward captured in a CUDA graph and replayed (GB300 only).  The library
neither allocates nor synchronises inside a call (the caller passes every buffer and the
workspace), so the calls are capturable; replays must reproduce the eager results."""
import math

import pytest
import torch

from bwd_xfa_fwd_gb300 import inputs
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bwd_xfa_fwd_gb300 import binding, build
    build.build()
    binding.load()
    assert torch.cuda.is_available()


# (dtype, hd, impl, bit-exact): the families without atomics replay bit for bit
CASES = [("f32", 64, 2, True), ("f32", 32, 2, True), ("bf16", 128, 3, True), ("bf16", 64, 3, True),
         ("bf16", 128, 2, False), ("f32", 64, 1, False)]


@pytest.mark.parametrize("dtype,hd,impl,exact", CASES)
def test_graph_replay_matches_eager(dtype, hd, impl, exact):
    from bwd_xfa_fwd_gb300 import binding
    bh, S = 3, 333
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), dtype, seed=88 + hd)
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    out = torch.empty_like(q)
    lse = torch.empty(bh, S, device="cuda", dtype=torch.float32)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    ws = torch.empty(binding.workspace_bytes(bh, S, hd, q.dtype), device="cuda", dtype=torch.uint8)

    def step():
        binding.fwd(q, k, v, scale, impl, out=out, lse=lse)
        binding.bwd(q, k, v, out, do, lse, scale, impl, workspace=ws, grads=grads)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, lse) + grads]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (out, lse) + grads:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert binding.status() == binding.XFA_OK
        for a, b in zip(eager, (out, lse) + grads):
            if exact:
                assert torch.equal(a, b)
            else:   # dQ summed with atomics in a data-dependent order (bf16: one rounding step apart)
                tol = (1e-2 if dtype == "bf16" else 1e-5) * float(a.float().abs().max())
                assert torch.allclose(a.float(), b.float(), rtol=0, atol=tol)


def test_concurrent_streams_and_counter_reuse():
    """The persistent tensor-core kernels take work items from a per-launch counter slot.  Forward
    and backward launches in flight on four streams at once, and more launches than there are
    slots (each slot resets itself when its launch ends), give the results of a lone launch."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd = 4, 1000, 128
    scale = 1.0 / math.sqrt(hd)
    cases = []
    for i in range(4):
        x = inputs.draw((bh, S, hd), "bf16", seed=300 + i)
        q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
        out, lse = binding.fwd(q, k, v, scale, binding.IMPL_TCGEN05_DET)
        grads = binding.bwd(q, k, v, out, do, lse, scale, binding.IMPL_TCGEN05_DET)
        torch.cuda.synchronize()
        cases.append(dict(qkvd=(q, k, v, do), ref=[t.clone() for t in (out, lse) + tuple(grads)]))
    streams = [torch.cuda.Stream() for _ in cases]
    for rep in range(20):   # 20 x 4 x 2 persistent launches: every counter slot is reused
        outs = []
        for c, st in zip(cases, streams):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                q, k, v, do = c["qkvd"]
                out, lse = binding.fwd(q, k, v, scale, binding.IMPL_TCGEN05_DET)
                grads = binding.bwd(q, k, v, out, do, lse, scale, binding.IMPL_TCGEN05_DET)
                outs.append((out, lse) + tuple(grads))
        torch.cuda.synchronize()
        assert binding.status() == binding.XFA_OK
        for c, o in zip(cases, outs):
            for a, b in zip(c["ref"], o):
                assert torch.equal(a, b), f"repetition {rep}"


def test_graph_replays_overlapping_eager_launches():
    """A captured launch keeps its work-counter slot for every replay; eager launches take
    theirs from another pool.  Replays of a captured forward + backward on one stream, with
    more eager launches than the eager pool has slots running on a second stream at the same
    time, both give the results of a lone launch."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd = 4, 1000, 128
    scale = 1.0 / math.sqrt(hd)
    impl = binding.IMPL_TCGEN05_DET
    cases = []
    for i in range(2):
        x = inputs.draw((bh, S, hd), "bf16", seed=700 + i)
        q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
        out, lse = binding.fwd(q, k, v, scale, impl)
        grads = binding.bwd(q, k, v, out, do, lse, scale, impl)
        torch.cuda.synchronize()
        cases.append(dict(qkvd=(q, k, v, do), ref=[t.clone() for t in (out, lse) + tuple(grads)]))
    q, k, v, do = cases[0]["qkvd"]
    out, lse = torch.empty_like(q), torch.empty(bh, S, device="cuda", dtype=torch.float32)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    ws = torch.empty(binding.workspace_bytes(bh, S, hd, q.dtype), device="cuda", dtype=torch.uint8)

    def step():
        binding.fwd(q, k, v, scale, impl, out=out, lse=lse)
        binding.bwd(q, k, v, out, do, lse, scale, impl, workspace=ws, grads=grads)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    replay_stream, eager_stream = torch.cuda.Stream(), torch.cuda.Stream()
    for t in (replay_stream, eager_stream):
        t.wait_stream(torch.cuda.current_stream())
    eager_outs = []
    for rep in range(70):   # 70 x 2 eager persistent launches: every eager slot is taken twice
        with torch.cuda.stream(replay_stream):
            g.replay()
        with torch.cuda.stream(eager_stream):
            qb, kb, vb, dob = cases[1]["qkvd"]
            ob, lb = binding.fwd(qb, kb, vb, scale, impl)
            gb = binding.bwd(qb, kb, vb, ob, dob, lb, scale, impl)
            if rep % 10 == 9:
                eager_outs.append((ob, lb) + tuple(gb))
        if rep % 10 == 9:
            replay_stream.synchronize()
            for a, b in zip(cases[0]["ref"], (out, lse) + grads):
                assert torch.equal(a, b), f"replay {rep}"
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    for o in eager_outs:
        for a, b in zip(cases[1]["ref"], o):
            assert torch.equal(a, b)


def test_graph_replays_the_cached_dropout_step():
    """The dropout step with its mask drawn by its own kernel and read by both attention kernels
    (xfa_dropout_keep_fill, xfa_fwd_dropout_cached, xfa_bwd_dropout_cached) captured once and
    replayed: every replay gives the eager results (dQ up to the order of its reduce-adds)."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd, p, seed = 3, 700, 128, 0.15, 0xD00D
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), "bf16", seed=91)
    q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
    out = torch.empty_like(q)
    lse = torch.empty(bh, S, device="cuda", dtype=torch.float32)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    ws = torch.empty(binding.workspace_bytes(bh, S, hd, q.dtype), device="cuda", dtype=torch.uint8)
    keep = torch.empty(binding.dropout_keep_bytes(bh, S), device="cuda", dtype=torch.uint8)

    def step():
        binding.dropout_keep_fill(bh, S, p, seed, keep, stream_of=q)
        binding.fwd(q, k, v, scale, out=out, lse=lse, dropout_p=p, keep_bits=keep, keep_cached=True)
        binding.bwd(q, k, v, out, do, lse, scale, workspace=ws, grads=grads, dropout_p=p, keep_bits=keep)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, lse) + grads]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (out, lse) + grads:
            t.fill_(float("nan"))
        keep.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert binding.status() == binding.XFA_OK
        for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), eager, (out, lse) + grads):
            if name == "dq":
                tol = 1e-2 * float(a.float().abs().max())
                assert torch.allclose(a.float(), b.float(), rtol=0, atol=tol), name
            else:
                assert torch.equal(a, b), name
