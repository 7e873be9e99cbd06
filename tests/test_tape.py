"""Tape engine semantics on CPU scalars, pinned to the worked examples of the pages."""
import json
import os

import torch

from bwd_xfa_fwd_gb300.tape import Var

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "value_tape_examples.json")


# test-only elementwise nodes (closures push grads to parents, as the tape expects)
def mul(a, b):
    return Var(a.value * b.value, (a, b), lambda g, ps: (ps[0].accumulate(g * ps[1].value),
                                                        ps[1].accumulate(g * ps[0].value)))


def add(a, b):
    return Var(a.value + b.value, (a, b), lambda g, ps: (ps[0].accumulate(g), ps[1].accumulate(g)))


def square(a):
    return Var(a.value ** 2, (a,), lambda g, ps: ps[0].accumulate(g * 2 * ps[0].value))


def leaf(x):
    return Var(torch.tensor(float(x), dtype=torch.float64))


def load():
    with open(GOLDEN) as f:
        return json.load(f)


def test_value_example_abc():
    g = load()["abc"]
    a, b, c = leaf(g["a"]), leaf(g["b"]), leaf(g["c"])
    L = square(add(mul(a, b), c))
    assert float(L.value) == g["L"]
    L.backward()
    assert float(a.grad) == g["grad"]["a"]
    assert float(b.grad) == g["grad"]["b"]
    assert float(c.grad) == g["grad"]["c"]


def test_value_example_xy_and_update():
    g = load()["xy"]
    x, y = leaf(g["x"]), leaf(g["y"])
    two = leaf(2.0)
    L = square(add(mul(x, y), two))
    assert float(L.value) == g["L"]
    L.backward()
    assert float(x.grad) == g["grad"]["x"] and float(y.grad) == g["grad"]["y"]
    assert abs(g["x"] - g["lr"] * float(x.grad) - g["updated"]["x"]) < 1e-12
    assert abs(g["y"] - g["lr"] * float(y.grad) - g["updated"]["y"]) < 1e-12


def test_fanout_accumulation_is_4x():
    factor = load()["fanout"]["factor"]
    xv = torch.tensor([0.5, -1.5, 2.0], dtype=torch.float64)
    x = Var(xv)
    y = add(mul(x, x), mul(x, x))
    y.backward()
    assert torch.equal(x.grad, factor * xv)


def test_topological_order_and_dedup():
    a = leaf(1.0)
    b = mul(a, a)
    c = add(b, b)
    order = c.topo_order()
    assert order[-1] is c and order[0] is a
    assert len(order) == len({id(n) for n in order}) == 3


def test_borrowed_grad_not_modified_in_place():
    # add() pushes the same upstream tensor to both parents; a later second push
    # into one parent must not change the other parent's gradient.
    x, z = leaf(1.0), leaf(2.0)
    s = add(x, z)
    t = add(s, x)          # x gets a second contribution
    t.backward()
    assert float(x.grad) == 2.0 and float(z.grad) == 1.0
