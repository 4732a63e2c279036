"""tp_attention_decode_noalloc: the decode-attention entry point for callers
that cannot allocate device memory on their decode path (code running in a
memory pool it does not own, a host framework that forbids cudaMalloc there,
a process whose allocator is exhausted).  It must give the same result as
tp_attention_heads with a caller-provided scratch buffer, on consecutive
calls that share its fixed device scratch array.

Kept in a file of its own, named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_fp32, np64
from tensor_transformer_layer_03_b300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(tp, d, H, deg, B, cap, dtype, seed):
    plan = tp.Plan(d, H, 8 * deg, deg, act="swiglu", dtype=dtype)
    dh = d // H
    g = torch.Generator().manual_seed(seed)
    tdt = I.torch_dtype(dtype)
    qkv = torch.stack([I.make_matrix(B, 3 * d // deg, dtype, g) for _ in range(deg)]).to(DEV)
    kc = torch.randn(B, H, cap, dh, generator=g).to(tdt).to(DEV)
    vc = torch.randn(B, H, cap, dh, generator=g).to(tdt).to(DEV)
    return plan, qkv, kc, vc


def _reference(tp, plan, qkv, kc, vc, B, cap, pos, deg, d, dtype):
    """The existing entry point with a caller-provided scratch buffer."""
    out = torch.empty(deg, B, d // deg, dtype=I.torch_dtype(dtype), device=DEV)
    scratch = torch.empty(plan.attention_scratch_bytes(B, 1, cap), dtype=torch.uint8, device=DEV)
    k2, v2 = kc.clone(), vc.clone()
    plan.attention_heads(qkv, B, 1, True, k2, v2, cap, pos, out, scratch)
    plan.sync_status()
    return out, k2, v2


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_matches_existing_entry_point_twice(tp, dtype):
    check = assert_close_bf16 if dtype == "bf16" else assert_close_fp32
    # two calls in a row on different shapes/positions: the second call must
    # not see anything the first one left in the shared scratch array
    for (d, H, deg, B, cap, pos, seed) in ((4096, 32, 2, 1, 1025, 1024, 1), (512, 8, 4, 3, 4000, 2999, 2)):
        plan, qkv, kc, vc = _case(tp, d, H, deg, B, cap, dtype, seed)
        ref, kref, vref = _reference(tp, plan, qkv, kc, vc, B, cap, pos, deg, d, dtype)
        out = torch.full((deg, B, d // deg), float("nan"), dtype=I.torch_dtype(dtype), device=DEV)
        k2, v2 = kc.clone(), vc.clone()
        plan.attention_decode_noalloc(qkv, B, k2, v2, cap, pos, out)
        plan.sync_status()
        check(out.cpu(), np64(ref.cpu()), f"noalloc d{d} B{B} pos{pos}")
        assert torch.equal(k2, kref) and torch.equal(v2, vref)
    # and the same call again: identical to its own first result
    out2 = torch.empty_like(out)
    k3, v3 = kc.clone(), vc.clone()
    plan.attention_decode_noalloc(qkv, B, k3, v3, cap, pos, out2)
    plan.sync_status()
    check(out2.cpu(), np64(ref.cpu()), "noalloc repeated call")


def test_noalloc_rejects_batches_beyond_its_scratch(tp):
    plan, qkv, kc, vc = _case(tp, 4096, 32, 2, 1, 8, "bf16", 3)
    out = torch.empty(2, 1, 2048, dtype=torch.bfloat16, device=DEV)
    # 8 MiB holds batch * 32 heads * 64 chunks * 130 floats for batch <= 7
    with pytest.raises(tp.TPError) as ei:
        plan.attention_decode_noalloc(qkv, 8, kc, vc, 8, 3, out)
    assert ei.value.name == "WORKSPACE_TOO_SMALL"
    plan.sync_status()
