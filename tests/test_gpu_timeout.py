"""Failure detection on the GPU without a fault: a bounded device wait that
runs out.

The tensor-core kernels never wait without a limit: every mbarrier wait and
every split-tile counter wait gives up after tp_set_wait_timeout_ns() of
%globaltimer, records an error word, raises the CTA's abort flag so the
other roles leave their loops, lets in-flight copies and tensor-core work
finish, frees its tensor memory and returns.  Here the limit is set to 1 ns
so that the first wait that is not satisfied at once runs out, on the
one-SM GEMM tiles (M <= 128); the call must still return, tp_sync_status
must report TP_ERR_DEVICE_TIMEOUT exactly once, and the next call on the
same plan and the same scratch must be correct (a launch that splits tiles
clears its own counters, so a timed-out one leaves nothing behind).  Nothing waits forever and no memory is touched out of bounds, so
the GPU context stays usable.
"""
import pytest
import torch

import oracle.tp_oracle as o
from helpers import assert_close_bf16, qkv_shards
from tensor_transformer_layer_03_b300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TP_ERR_DEVICE_TIMEOUT = 11


def _status(tp):
    return tp.tp_sync_status(tp._stream(None))


def test_gemm_wait_runs_out_and_recovers(tp):
    d, H, f, deg, M = 4096, 32, 11008, 2, 64
    plan = tp.Plan(d, H, f, deg)
    g = torch.Generator().manual_seed(41)
    w = I.make_weights(I.BlockShape(d, H, f, "swiglu"), "bf16", g)
    pw, _ = plan.sizes(1, 1)
    packed = torch.empty(pw, dtype=torch.uint8, device=DEV)
    plan.shard_weights({k: v.to(DEV) for k, v in w.items()}, packed)
    x = I.make_matrix(M, d, "bf16", g)
    xd = x.to(DEV)
    out = torch.zeros(deg, M, 3 * d // deg, dtype=torch.bfloat16, device=DEV)
    scr = torch.zeros(plan.linear_scratch_bytes(M), dtype=torch.uint8, device=DEV)
    assert plan.linear_schedule(0, tp.TP_QKV, M, scr.numel()).kernel == 0  # the tensor-core GEMM
    assert _status(tp) == 0
    tp.tp_set_wait_timeout_ns(1)
    try:
        plan.column_linear(tp.TP_QKV, xd, M, packed, out, scratch=scr)
        code = _status(tp)
    finally:
        tp.tp_set_wait_timeout_ns(0)  # back to the default limit
    assert code == TP_ERR_DEVICE_TIMEOUT, tp.status_name(code)
    assert _status(tp) == 0  # reported once, then cleared
    # the context is usable and the plan works again, on the same scratch
    plan.column_linear(tp.TP_QKV, xd, M, packed, out, scratch=scr)
    assert _status(tp) == 0
    ref = qkv_shards(o.linear(x, w["Wq"]), o.linear(x, w["Wk"]), o.linear(x, w["Wv"]), deg, H)
    assert_close_bf16(out.cpu(), o.round_bf16(ref), "QKV after a timed-out launch")
