"""GPU parity of the sequence-parallel calls (token rows held as tp slices
around the tensor-parallel regions: reduce-scatter after the row-parallel
linears, all-gather before the column-parallel ones) against the float64
oracle's sequence_parallel_block_forward, and bit for bit against the plain
calls on the same rows (the same tiles and sums, only the rows' addresses
differ).  Slices sit in padded regions; the padding must stay untouched."""
import pytest
import torch

import oracle.tp_oracle as o
from helpers import BF16_MEAN_ABS, FLOOR_FACTOR, assert_close_bf16, mean_abs, np64
from tensor_transformer_layer_03_b300 import inputs as I
from tensor_transformer_layer_03_b300.runtime import TPBlock

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAD = 24  # extra rows per slice region


def _slices(rows, tp, pad, dtype, fill=0.0):
    """[M, d] -> [tp][M/tp + pad][d] with the slice in the first M/tp rows."""
    M, d = rows.shape
    ms = M // tp
    out = torch.full((tp, ms + pad, d), fill, dtype=dtype)
    for s in range(tp):
        out[s, :ms] = rows[s * ms:(s + 1) * ms]
    return out


def _unslice(t, M):
    tp = t.shape[0]
    ms = M // tp
    return torch.cat([t[s, :ms] for s in range(tp)], dim=0)


@pytest.mark.parametrize("deg", [2, 4, 8])
@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_block_forward_seq(tp, deg, act):
    shape = I.BlockShape(1024, 8, 2816, act)
    wl = I.Workload("seq", shape, tp=deg, batch=2, seq=128, causal=True, dtype="bf16")
    inp = I.make_inputs(wl, seed=11)
    w = {n: v for n, v in inp.items() if n.startswith("W")}
    B, T, d = wl.batch, wl.seq, shape.d_model
    M = B * T
    blk = TPBlock(shape, deg, "bf16", w, device=DEV, max_batch=B, max_seq=T)
    xs = _slices(inp["X"].reshape(M, d), deg, PAD, torch.bfloat16).to(DEV)
    ys = torch.full((deg, M // deg + PAD, d), float("nan"), dtype=torch.float32, device=DEV)
    blk.forward_seq(xs, B, T, True, out_slices=ys)
    blk.plan.sync_status()
    y_plain = blk.forward(inp["X"].to(DEV), True).reshape(M, d)
    blk.plan.sync_status()
    ysc = ys.cpu()
    assert torch.isnan(ysc[:, M // deg:]).all(), "padding rows of the output slices were written"
    got = _unslice(ysc, M)
    assert torch.equal(got, y_plain.cpu()), "sequence-parallel block differs from the plain block"
    ex, ysl, _ = o.sequence_parallel_block_forward(inp["X"], w, shape.n_heads, act, True, deg)
    st, _, _ = o.block_forward(inp["X"], w, shape.n_heads, act, True, storage="bf16")
    floor = mean_abs(st, ex)
    assert_close_bf16(got.reshape(B, T, d), ex, f"seq block tp{deg} {act}",
                      mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * floor))
    # slice s of the output is the oracle's slice s
    for s in range(deg):
        assert_close_bf16(ysc[s, :M // deg], ysl[s], f"slice {s}", mean_abs_bound=max(BF16_MEAN_ABS, 1.5 * floor))


def test_block_forward_seq_prenorm(tp):
    """Pre-norm plan: the RMSNorm of x runs on the slices' rows."""
    shape, deg, B, T, eps, theta = I.BlockShape(512, 8, 1536, "swiglu"), 4, 1, 256, 1e-5, 10000.0
    g = torch.Generator().manual_seed(12)
    w = I.make_weights(shape, "bf16", g)
    w.update(I.make_norm_gains(shape, "bf16", g))
    x = torch.randn(B, T, shape.d_model, generator=g).to(torch.bfloat16)
    M, d = B * T, shape.d_model
    blk = TPBlock(shape, deg, "bf16", w, device=DEV, max_batch=B, max_seq=T, rms_eps=eps, rope_theta=theta)
    xs = _slices(x.reshape(M, d), deg, PAD, torch.bfloat16).to(DEV)
    ys = blk.forward_seq(xs, B, T, True)
    y_plain = blk.forward(x.to(DEV), True).reshape(M, d)
    blk.plan.sync_status()
    got = _unslice(ys.cpu(), M)
    assert torch.equal(got, y_plain.cpu())
    ex, _, _ = o.llama_block_forward(x, w, shape.n_heads, True, eps, theta)
    st, _, _ = o.llama_block_forward(x, w, shape.n_heads, True, eps, theta, storage="bf16")
    assert_close_bf16(got.reshape(B, T, d), ex, "seq pre-norm block",
                      mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * mean_abs(st, ex)))


@pytest.mark.parametrize("deg,M", [(4, 2048), (2, 256), (8, 128)])
def test_gather_and_reduce_scatter_calls(tp, deg, M):
    """The per-call forms at the 7B shape: column linears reading gathered
    slices and row-parallel linears writing their rows (plus the residual's)
    into slices give the plain calls' bits."""
    d, H, f = 4096, 32, 11008
    plan = tp.Plan(d, H, f, deg)
    shape = I.BlockShape(d, H, f, "swiglu")
    g = torch.Generator().manual_seed(13)
    w = I.make_weights(shape, "bf16", g)
    pw, _ = plan.sizes(1, 1)
    packed = torch.empty(pw, dtype=torch.uint8, device=DEV)
    plan.shard_weights({k: v.to(DEV) for k, v in w.items()}, packed)
    scr = torch.zeros(max(plan.linear_scratch_bytes(M), 16), dtype=torch.uint8, device=DEV)
    ms, cap = M // deg, M // deg + PAD
    x = I.make_matrix(M, d, "bf16", g)
    xs = _slices(x, deg, PAD, torch.bfloat16).to(DEV)
    for which, n_out in ((tp.TP_QKV, 3 * d // deg), (tp.TP_FFN_UP, f // deg)):
        a = torch.empty(deg, M, n_out, dtype=torch.bfloat16, device=DEV)
        b = torch.empty_like(a)
        plan.column_linear(which, x.to(DEV), M, packed, a, scratch=scr)
        plan.column_linear_gather(which, xs, cap * d, M, packed, b, scratch=scr)
        plan.sync_status()
        assert torch.equal(a, b), which
    for which, ks, res_dtype in ((tp.TP_ATTN_OUT, d // deg, "bf16"), (tp.TP_FFN_DOWN, f // deg, "fp32")):
        inp = torch.stack([I.make_matrix(M, ks, "bf16", g) for _ in range(deg)]).to(DEV)
        res = I.make_matrix(M, d, res_dtype, g)
        tdt = I.torch_dtype(res_dtype)
        out, act = torch.empty(M, d, device=DEV), torch.empty(M, d, dtype=torch.bfloat16, device=DEV)
        plan.row_linear_reduce(which, inp, M, packed, res.to(DEV), out, act, scratch=scr)
        # the residual and both outputs as slices of one stride (residual in its own dtype's elements)
        rs = _slices(res, deg, PAD, tdt).to(DEV)
        outs = torch.full((deg, cap, d), float("nan"), device=DEV)
        acts = torch.full((deg, cap, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        plan.row_linear_reduce_scatter(which, inp, M, packed, rs, outs, acts, cap * d, scratch=scr)
        plan.sync_status()
        assert torch.equal(_unslice(outs, M), out) and torch.equal(_unslice(acts, M), act), which
        assert torch.isnan(outs[:, ms:]).all() and torch.isnan(acts[:, ms:].float()).all()
