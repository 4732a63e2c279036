"""GPU parity of batched, multi-step decode with a growing KV cache.

n single-token steps at cache positions P, P+1, ..., P+n-1 (each step's K/V
appended by the library and read back by the later steps) must equal one
oracle pass of the n tokens over the P-position prefix with the causal mask:
token i at position P+i attends to the prefix and to tokens 0..i.  Bounds as
in test_gpu_block.py (normwise <= 2e-2 against the exact oracle, mean abs
against the oracle's bf16-storage floor)."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as o
from helpers import BF16_MEAN_ABS, FLOOR_FACTOR, assert_close_bf16, mean_abs
from tensor_transformer_layer_03_b300 import inputs as I
from tensor_transformer_layer_03_b300.runtime import TPBlock

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _decode_steps(shape, deg, B, P, n, seed):
    """Returns (GPU outputs [B, n, d], exact oracle, bf16-storage oracle,
    GPU cache rows P..P+n-1 of K, oracle K of the n tokens)."""
    wl = I.Workload("decode_steps", shape, tp=deg, batch=B, seq=n, causal=True, dtype="bf16", decode=True,
                    cache_len=P)
    inp = I.make_inputs(wl, seed=seed)
    w = {k: v for k, v in inp.items() if k.startswith("W")}
    H, dh = shape.n_heads, shape.d_head
    cap = P + n + 3  # room past the last step: must stay untouched
    kc = torch.full((B, H, cap, dh), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, H, cap, dh), float("nan"), dtype=torch.bfloat16)
    kc[:, :, :P] = inp["Kcache"]
    vc[:, :, :P] = inp["Vcache"]
    kd, vd = kc.to(DEV), vc.to(DEV)
    blk = TPBlock(shape, deg, "bf16", w, device=DEV, max_batch=B, max_seq=1)
    x = inp["X"].to(DEV)
    ys = []
    for i in range(n):
        ys.append(blk.forward(x[:, i:i + 1].contiguous(), True, k_cache=kd, v_cache=vd, cache_pos=P + i).cpu())
    blk.plan.sync_status()
    got = torch.cat(ys, dim=1)
    ex, K, _ = o.block_forward(inp["X"], w, H, shape.act, True, kcache=kc, vcache=vc, cache_pos=P)
    st, _, _ = o.block_forward(inp["X"], w, H, shape.act, True, kcache=kc, vcache=vc, cache_pos=P, storage="bf16")
    kn = kd.cpu()
    assert torch.isnan(kn[:, :, P + n:]).all(), "cache rows past the last step were written"
    return got, ex, st, kn[:, :, P:P + n], K


@pytest.mark.parametrize("B,shape,deg,P,n", [
    (4, I.BlockShape(1024, 8, 2816, "swiglu"), 2, 200, 6),    # weight-streaming linears (M <= 4)
    (8, I.BlockShape(1024, 8, 2816, "swiglu"), 2, 90, 3),     # tensor-core weight stream, 8 rows
    (16, I.BlockShape(1024, 8, 2816, "swiglu"), 2, 130, 5),   # tensor-core weight stream, 2 groups of 8 rows
    (24, I.BlockShape(1024, 8, 2816, "swiglu"), 2, 60, 2),    # tensor-core weight stream, 4 groups (ragged)
    (64, I.BlockShape(512, 4, 1536, "swiglu"), 4, 70, 3),     # tensor-core GEMM, split tiles of one m-block
])
def test_multistep_decode_growing_cache(tp, B, shape, deg, P, n):
    got, ex, st, k_gpu, k_ref = _decode_steps(shape, deg, B, P, n, seed=11)
    floor = mean_abs(st, ex)
    assert_close_bf16(got, ex, f"{n}-step decode B={B}", mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * floor))
    # every appended K row is the bf16 value of that step's projection
    assert_close_bf16(k_gpu, o.round_bf16(k_ref), "appended K rows")


def test_llama7b_decode_batch16(tp):
    """The 7B-shaped decode workload with 16 sequences (the tensor-core
    weight stream with two groups of 8 token rows), one step over 1024
    cached positions."""
    shape = I.LLAMA7B
    got, ex, st, _, _ = _decode_steps(shape, 2, 16, 1024, 1, seed=0)
    floor = mean_abs(st, ex)
    assert_close_bf16(got, ex, "7B decode B=16", mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * floor))
