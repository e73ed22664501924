"""Host logic of the prequantized expert-weight cache (no GPU): a cached quadruple is reused
across microbatches while the weight is unchanged and dropped when it changes in place, is
replaced, or the optimizer steps ("feat(moe): add MoK MXFP8 expert support", Summary: the
prequantized-weight cache retained across microbatches until the optimizer step)."""
import gc

import torch

from mxfp8_precision_moe_gb300.weight_cache import Mxfp8WeightCache


class FakeQuantize:
    """Stands in for the GPU quantization: records calls, returns fresh tensors."""

    def __init__(self):
        self.calls = 0

    def __call__(self, W):
        self.calls += 1
        G, N, K = W.shape
        return (torch.full((G, N, K), self.calls, dtype=torch.uint8), torch.zeros(G, 1, dtype=torch.uint8),
                torch.full((G, K, N), self.calls, dtype=torch.uint8), torch.zeros(G, 1, dtype=torch.uint8))


def make():
    fq = FakeQuantize()
    return fq, Mxfp8WeightCache(quantize=fq)


def test_reused_across_microbatches():
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    quads = [cache.get(W) for _ in range(4)]
    assert fq.calls == 1 and cache.misses == 1 and cache.hits == 3
    assert all(q is quads[0] for q in quads)


def test_in_place_update_invalidates():
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    q0 = cache.get(W)
    with torch.no_grad():
        W.add_(1.0)                      # bumps the version counter
    q1 = cache.get(W)
    assert fq.calls == 2 and q1 is not q0
    assert int(q0[0][0, 0, 0]) == 1 and int(q1[0][0, 0, 0]) == 2  # the old quadruple is untouched


def test_optimizer_step_invalidates():
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    opt = torch.optim.SGD([W], lr=0.1)
    handle = cache.attach(opt)
    cache.get(W)
    cache.get(W)
    W.grad = torch.ones_like(W)
    opt.step()
    assert len(cache) == 0
    cache.get(W)
    assert fq.calls == 2
    handle.remove()


def test_data_write_needs_the_optimizer_hook():
    # a write through .data does not bump the parameter's version: the cache only sees it
    # through invalidate() (which attach() calls after each optimizer step)
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    cache.get(W)
    W.data.mul_(2.0)
    cache.get(W)
    assert fq.calls == 1
    cache.invalidate()
    cache.get(W)
    assert fq.calls == 2


def test_replaced_storage_and_shape_invalidate():
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    cache.get(W)
    W.data = torch.randn(2, 4, 8, dtype=torch.bfloat16)   # new storage, same object
    cache.get(W)
    assert fq.calls == 2
    W.data = torch.randn(2, 8, 8, dtype=torch.bfloat16)   # new shape
    q = cache.get(W)
    assert fq.calls == 3 and q[0].shape == (2, 8, 8)


def test_distinct_weights_have_distinct_entries():
    fq, cache = make()
    Wg = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    Wu = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    a, b = cache.get(Wg), cache.get(Wu)
    assert a is not b and fq.calls == 2
    assert cache.get(Wg) is a and cache.get(Wu) is b and fq.calls == 2


def test_dead_weight_is_not_matched():
    # a new tensor that reuses a freed tensor's id (and possibly its address) must not hit
    fq, cache = make()
    W = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    cache.get(W)
    del W
    gc.collect()
    assert len(cache) == 0
    W2 = torch.nn.Parameter(torch.randn(2, 4, 8, dtype=torch.bfloat16))
    cache.get(W2)
    assert fq.calls == 2
