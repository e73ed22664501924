"""Prequantized expert-weight cache.

"feat(moe): add MoK MXFP8 expert support" (Summary; review of the ``mxfp8_weights`` argument):
the routed-expert weights are quantized to MXFP8 once and the result is kept, per layer, across
the microbatches of one optimizer step; the backward takes the same quadruple
``(weight_fp8, weight_scale, weight_t_fp8, weight_t_scale)``.  The plain pair feeds the forward
GEMM (scales along K), the transposed pair the dgrad GEMM (scales along N).

A cached quadruple is reused while the weight is provably unchanged: the same tensor object
(held by weak reference), the same storage pointer, offset, shape, stride and dtype, and the
same in-place version counter (an optimizer that updates the parameter in place bumps it).
Optimizers that write through ``.data`` do not bump the version, so ``attach(optimizer)``
also drops every entry after each ``optimizer.step()``.  A refill allocates new tensors and
never writes into a quadruple handed out earlier, so tensors saved for a pending backward stay
valid.
"""
from __future__ import annotations

import weakref
from typing import Callable, Optional

import torch

Quad = tuple  # (weight_fp8 [G,N,K], weight_scale, weight_t_fp8 [G,K,N], weight_t_scale)


def _stamp(W: torch.Tensor) -> tuple:
    return (W.device, W.untyped_storage().data_ptr(), W.storage_offset(), tuple(W.shape), tuple(W.stride()),
            W.dtype, W._version)


class Mxfp8WeightCache:
    """Per-layer cache of MXFP8 expert weights, valid until the weight changes or the
    optimizer steps.

    ``quantize(W) -> quad`` defaults to one fused plain + transposed quantization of
    ``W[G, N, K]`` into blocked scales (``quantize_expert_weights``; with ``block32x32``,
    one scale per 32x32 block).  ``hits`` and ``misses`` count lookups."""

    def __init__(self, quantize: Optional[Callable[[torch.Tensor], Quad]] = None, block32x32: bool = False):
        if quantize is None:
            from . import quantize_expert_weights

            quantize = lambda W: quantize_expert_weights(W, block32x32=block32x32)  # noqa: E731
        self._quantize = quantize
        self._entries: dict[int, tuple] = {}  # id(W) -> (weakref(W), stamp, quad)
        self.hits = 0
        self.misses = 0

    def get(self, W: torch.Tensor) -> Quad:
        """The quadruple for W: cached if W is unchanged since it was quantized, else a new one."""
        key = id(W)
        ent = self._entries.get(key)
        stamp = _stamp(W)
        if ent is not None and ent[0]() is W and ent[1] == stamp:
            self.hits += 1
            return ent[2]
        quad = self._quantize(W)
        self.misses += 1
        self._entries[key] = (weakref.ref(W), stamp, quad)
        return quad

    def invalidate(self) -> None:
        """Drop every cached quadruple (the next ``get`` quantizes again)."""
        self._entries.clear()

    def __len__(self) -> int:
        return sum(1 for ref, _, _ in self._entries.values() if ref() is not None)

    def attach(self, optimizer: torch.optim.Optimizer):
        """Invalidate after every ``optimizer.step()``; returns the hook handle."""
        return optimizer.register_step_post_hook(lambda *args, **kwargs: self.invalidate())
