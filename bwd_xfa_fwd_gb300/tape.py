"""A minimal define-by-run tape and the fused flash-attention node on it.

Tape semantics follow "xtrain docs/03-autograd-engine.md", section
"Tape 设计：Rc<RefCell<VarNode>> + 逆拓扑遍历" and "梯度累加（扇出求和）":
a ``Var`` holds a value, an optional gradient, its parents and a backward
closure ``fn(grad, parents)``; ``backward()`` builds a post-order DFS
topological order (deduplicated by identity), seeds the output gradient with
ones and walks the order in reverse, each closure pushing gradient
contributions to its parents; every push sums into the existing gradient, so
fan-out (one Var consumed several times, even twice by the same node) is
correct.

``flash_attention(q, k, v)`` is the operator of "xtrain docs/13-flash-attention.md"
as one node (sections "Module Layout" and design decision ②): the forward
runs ``xfa_fwd`` and the node keeps only the O(N) logsumexp L (plus its
parents and O); the backward runs ``xfa_bwd``.  Gradient sums on CUDA tensors
use the library's ``xfa_accumulate`` kernel.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch


class Var:
    __slots__ = ("value", "grad", "parents", "backward_fn", "saved", "_grad_owned", "__weakref__")

    def __init__(self, value: torch.Tensor, parents: Sequence["Var"] = (),
                 backward_fn: Optional[Callable[[torch.Tensor, Sequence["Var"]], None]] = None):
        self.value = value
        self.grad: Optional[torch.Tensor] = None
        self.parents = tuple(parents)
        self.backward_fn = backward_fn   # None for a leaf
        self.saved = {}                  # what a node keeps for its backward
        self._grad_owned = False         # False while self.grad may alias another node's tensor

    def accumulate(self, g: torch.Tensor) -> None:
        """Sum a gradient contribution into ``self.grad`` (first push stores it)."""
        if self.grad is None:
            self.grad = g
            self._grad_owned = False
            return
        if not self._grad_owned:           # never add in place into a borrowed tensor
            self.grad = self.grad.clone()
            self._grad_owned = True
        if g.is_cuda and g.dtype in (torch.float32, torch.bfloat16) and g.shape == self.grad.shape:
            from . import binding
            binding.accumulate_(self.grad, g.contiguous())
        else:
            self.grad += g

    def topo_order(self):
        """Post-order DFS from this node; each node once (by identity)."""
        order, seen = [], set()
        stack = [(self, False)]
        while stack:
            node, expanded = stack.pop()
            if expanded:
                order.append(node)
                continue
            if id(node) in seen:
                continue
            seen.add(id(node))
            stack.append((node, True))
            for p in reversed(node.parents):
                if id(p) not in seen:
                    stack.append((p, False))
        return order

    def backward(self, seed: Optional[torch.Tensor] = None) -> None:
        """Reverse-mode sweep from this node; the seed defaults to ones."""
        order = self.topo_order()
        self.grad = torch.ones_like(self.value) if seed is None else seed
        for node in reversed(order):
            if node.backward_fn is not None and node.grad is not None:
                node.backward_fn(node.grad, node.parents)

    def __repr__(self):
        return f"Var(shape={tuple(self.value.shape)}, dtype={self.value.dtype}, leaf={self.backward_fn is None})"


def flash_attention(q: Var, k: Var, v: Var, scale: Optional[float] = None, impl: int = 0, dropout_p: float = 0.0,
                    seed: int = 0, keep_mask: bool = False) -> Var:
    """Causal flash attention as one tape node: returns Var(O); caches L.  ``dropout_p`` > 0
    drops attention probabilities with the counter-based mask of ``seed``; the backward
    re-draws the same mask (nothing but the seed is kept), or, with ``keep_mask`` (bf16
    tensor-core kernels), reads the mask the forward stored as bits (bh * S^2 / 8 bytes kept
    with the node) instead of drawing it again."""
    from . import binding

    keep = None
    if dropout_p and keep_mask:
        bh, S, _ = binding._shape3(q.value)
        keep = torch.empty(binding.dropout_keep_bytes(bh, S), device=q.value.device, dtype=torch.uint8)
    out, lse = binding.fwd(q.value, k.value, v.value, scale, impl, dropout_p=dropout_p, seed=seed, keep_bits=keep)
    hd = q.value.shape[-1]
    sc = binding.default_scale(hd) if scale is None else float(scale)

    def backward_fn(grad, parents):
        pq, pk, pv = parents
        dq, dk, dv = binding.bwd(pq.value, pk.value, pv.value, out, grad.contiguous(), lse, sc, impl,
                                 dropout_p=dropout_p, seed=seed, keep_bits=keep)
        pq.accumulate(dq)
        pk.accumulate(dk)
        pv.accumulate(dv)

    node = Var(out, (q, k, v), backward_fn)
    node.saved["lse"] = lse
    if keep is not None:
        node.saved["keep_bits"] = keep
    return node
