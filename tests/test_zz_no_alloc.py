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

import oracle.tp_oracle as o
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


def _oracle_decode(qkv, kc, vc, pos, deg, H):
    """Float64 oracle of the one-token attention: shard s, local head j
    (global head s * H / deg + j) attends over its cached keys 0..pos-1 and
    the new token's key at pos."""
    qkv, kc, vc = np64(qkv.cpu()), np64(kc.cpu()), np64(vc.cpu())
    hl = H // deg
    dh = qkv.shape[2] // (3 * hl)
    out = np.zeros((deg, qkv.shape[1], hl * dh))
    for s in range(deg):
        for b in range(qkv.shape[1]):
            for j in range(hl):
                h = s * hl + j
                q = qkv[s, b, j * dh:(j + 1) * dh]
                kn = qkv[s, b, (hl + j) * dh:(hl + j + 1) * dh]
                vn = qkv[s, b, (2 * hl + j) * dh:(2 * hl + j + 1) * dh]
                keys = np.concatenate([kc[b, h, :pos], kn[None]], axis=0)
                vals = np.concatenate([vc[b, h, :pos], vn[None]], axis=0)
                out[s, b, j * dh:(j + 1) * dh] = o.attention_head(q[None], keys, vals, False)[0]
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_matches_existing_entry_point_twice(tp, dtype):
    check = assert_close_bf16 if dtype == "bf16" else assert_close_fp32
    # calls in a row on different shapes/positions: a call must not see
    # anything an earlier one left in the shared scratch array.  The long
    # caches take the routes with a separate append (bf16 past 4096
    # positions) and with capped splits (past 8192 positions).
    cases = [(4096, 32, 2, 1, 1025, 1024, 1), (512, 8, 4, 3, 4000, 2999, 2), (512, 8, 2, 2, 5000, 4500, 4)]
    if dtype == "fp32":
        cases.append((256, 4, 2, 1, 9000, 8500, 5))
    for (d, H, deg, B, cap, pos, seed) in cases:
        plan, qkv, kc, vc = _case(tp, d, H, deg, B, cap, dtype, seed)
        ref, kref, vref = _reference(tp, plan, qkv, kc, vc, B, cap, pos, deg, d, dtype)
        out = torch.full((deg, B, d // deg), float("nan"), dtype=I.torch_dtype(dtype), device=DEV)
        k2, v2 = kc.clone(), vc.clone()
        plan.attention_decode_noalloc(qkv, B, k2, v2, cap, pos, out)
        plan.sync_status()
        check(out.cpu(), np64(ref.cpu()), f"noalloc d{d} B{B} pos{pos}")
        assert torch.equal(k2, kref) and torch.equal(v2, vref)
        # and against the float64 oracle directly (bf16 output: the oracle
        # rounded to the storage type)
        ex = _oracle_decode(qkv, kc, vc, pos, deg, H)
        check(out.cpu(), o.round_bf16(ex) if dtype == "bf16" else ex, f"noalloc vs oracle d{d} pos{pos}")
    # and the same call again: bit for bit its own first result
    out2 = torch.empty_like(out)
    k3, v3 = kc.clone(), vc.clone()
    plan.attention_decode_noalloc(qkv, B, k3, v3, cap, pos, out2)
    plan.sync_status()
    assert torch.equal(out2, out), "noalloc repeated call differs"


def test_noalloc_rejects_batches_beyond_its_scratch(tp):
    plan, qkv, kc, vc = _case(tp, 4096, 32, 2, 1, 8, "bf16", 3)
    out = torch.empty(2, 1, 2048, dtype=torch.bfloat16, device=DEV)
    # 8 MiB holds batch * 32 heads * 64 chunks * 130 floats for batch <= 7
    with pytest.raises(tp.TPError) as ei:
        plan.attention_decode_noalloc(qkv, 8, kc, vc, 8, 3, out)
    assert ei.value.name == "WORKSPACE_TOO_SMALL"
    plan.sync_status()
