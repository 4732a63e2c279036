"""GPU parity of a stack of tensor-parallel blocks (tp_stack_forward)
against the float64 oracle's stack_forward: prefill, and multi-step decode
with one growing KV cache per layer.  The inter-layer activation is the
plan-dtype (bf16) copy of each layer's output in both.  Bounds as in
test_gpu_block.py: normwise <= 2e-2 against the exact oracle, mean abs
against the oracle's bf16-storage floor."""
import pytest
import torch

import oracle.tp_oracle as o
from helpers import BF16_MEAN_ABS, FLOOR_FACTOR, assert_close_bf16, mean_abs
from tensor_transformer_layer_03_b300 import inputs as I
from tensor_transformer_layer_03_b300.runtime import TPStack

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _layers(shape, n, seed):
    g = torch.Generator().manual_seed(seed)
    return [I.make_weights(shape, "bf16", g) for _ in range(n)], g


def _check(got, ex, st, what):
    floor = mean_abs(st, ex)
    assert_close_bf16(got, ex, what, mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * floor))


@pytest.mark.parametrize("shape,deg,L,B,T", [
    (I.BlockShape(512, 8, 1536, "swiglu"), 4, 3, 2, 160),
    (I.BlockShape(1024, 8, 2816, "swiglu"), 2, 4, 1, 300),
])
def test_stack_prefill(tp, shape, deg, L, B, T):
    layers, g = _layers(shape, L, 21)
    x = torch.randn(B, T, shape.d_model, generator=g).to(torch.bfloat16)
    stk = TPStack(shape, deg, "bf16", layers, device=DEV, max_batch=B, max_seq=T)
    y = stk.forward(x.to(DEV), True).cpu()
    stk.plan.sync_status()
    ex, _, _ = o.stack_forward(x, layers, shape.n_heads, shape.act, True)
    st, _, _ = o.stack_forward(x, layers, shape.n_heads, shape.act, True, storage="bf16")
    _check(y, ex, st, f"{L}-layer stack prefill")


def test_stack_multistep_decode(tp):
    """Per-layer caches with a random 90-position prefix, then 4 decode steps
    through the whole stack; step i equals row i of one oracle pass of the 4
    tokens at positions 90..93."""
    shape, deg, L, B, P, n = I.BlockShape(512, 4, 1536, "swiglu"), 2, 3, 4, 90, 4
    layers, g = _layers(shape, L, 22)
    H, dh = shape.n_heads, shape.d_head
    x = torch.randn(B, n, shape.d_model, generator=g).to(torch.bfloat16)
    kcs = [torch.randn(B, H, P + n, dh, generator=g).to(torch.bfloat16) for _ in range(L)]
    vcs = [torch.randn(B, H, P + n, dh, generator=g).to(torch.bfloat16) for _ in range(L)]
    kd = [k.to(DEV) for k in kcs]
    vd = [v.to(DEV) for v in vcs]
    stk = TPStack(shape, deg, "bf16", layers, device=DEV, max_batch=B, max_seq=1)
    xd = x.to(DEV)
    ys = [stk.forward(xd[:, i:i + 1].contiguous(), True, k_caches=kd, v_caches=vd, cache_pos=P + i).cpu()
          for i in range(n)]
    stk.plan.sync_status()
    got = torch.cat(ys, dim=1)
    ex, K, _ = o.stack_forward(x, layers, H, shape.act, True, kcs, vcs, P)
    st, _, _ = o.stack_forward(x, layers, H, shape.act, True, kcs, vcs, P, storage="bf16")
    _check(got, ex, st, f"{L}-layer stack, {n} decode steps")
    # each layer's cache got that layer's keys of the new tokens (the first
    # layer's inputs are exact, so its K matches the exact oracle at bf16)
    assert_close_bf16(kd[0][:, :, P:P + n].cpu(), o.round_bf16(K[0]), "layer-0 appended K")
