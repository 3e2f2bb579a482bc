"""Whole-tensor comparison of a GPU result with the fp64 oracle at full size.

The oracle runs on blocks of (b, h) sequences so that the fp64 copies of one
block stay near ``budget`` bytes; the squared differences and squared
reference norms are summed over every block, so the figure returned is the
relative Frobenius error ||x - x_ref||_F / ||x_ref||_F over the whole tensor,
the same number as one oracle call over everything would give.
"""
from __future__ import annotations

import numpy as np
import torch

SEQ_NAMES = ("q", "k", "v", "g", "beta")


def head_blocks(B: int, T: int, H: int, width: int, budget: int = 1 << 29):
    """(b, h0, h1) blocks covering every sequence; about ``budget`` bytes per
    fp64 input of a block (``width`` = the widest feature dimension)."""
    per_head = max(1, T * width * 8)
    hg = max(1, min(H, budget // per_head))
    for b in range(B):
        for h0 in range(0, H, hg):
            yield b, h0, min(H, h0 + hg)


def block_inputs(x: dict, b: int, h0: int, h1: int, extra: dict | None = None) -> dict:
    """The inputs of sequences (b, h0:h1) as a [1, T, h1-h0, *] problem."""
    sub = {n: x[n][b:b + 1, :, h0:h1].contiguous() for n in SEQ_NAMES}
    s0 = x.get("h0")
    sub["h0"] = None if s0 is None else s0[b:b + 1, h0:h1].contiguous()
    for n, t in (extra or {}).items():
        sub[n] = t[b:b + 1, :, h0:h1].contiguous()
    return sub


class Frobenius:
    """Accumulates ||got - ref||^2 and ||ref||^2 block by block."""

    def __init__(self):
        self.d2 = 0.0
        self.r2 = 0.0

    def add(self, got, ref):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        self.d2 += float(np.sum((got - ref) ** 2))
        self.r2 += float(np.sum(ref ** 2))

    @property
    def rel(self) -> float:
        return float(np.sqrt(self.d2) / (np.sqrt(self.r2) if self.r2 > 0 else 1.0))


def whole_errors(x: dict, o: torch.Tensor, hf: torch.Tensor | None, oracle, *, extra=None,
                 budget: int = 1 << 29):
    """Relative Frobenius errors of o (and h_final) over the whole tensors.

    ``oracle(sub) -> (o_ref, hf_ref)`` runs on one block's inputs (see
    ``block_inputs``); ``o`` [B,T,H,V] and ``hf`` [B,H,K,V] are the GPU results
    (any device). Every output must also be finite."""
    B, T, H, K = x["q"].shape
    V = x["v"].shape[-1]
    o_cpu = o.detach().cpu()
    hf_cpu = None if hf is None else hf.detach().cpu()
    assert torch.isfinite(o_cpu).all()
    if hf_cpu is not None:
        assert torch.isfinite(hf_cpu).all()
    eo, eh = Frobenius(), Frobenius()
    for b, h0, h1 in head_blocks(B, T, H, max(K, V), budget):
        sub = block_inputs(x, b, h0, h1, extra)
        o_ref, hf_ref = oracle(sub)
        eo.add(o_cpu[b:b + 1, :, h0:h1].double().numpy(), o_ref)
        if hf_cpu is not None:
            eh.add(hf_cpu[b:b + 1, h0:h1].double().numpy(), hf_ref)
    return eo.rel, (eh.rel if hf_cpu is not None else None)
