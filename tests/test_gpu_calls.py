"""GPU parity of each C-ABI call against the float64 oracle, on identical
seeded inputs.  bf16 outputs are compared with the oracle rounded to bf16
(the output's storage type); fp32 outputs with the exact oracle."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as o
from helpers import (assert_close_bf16, assert_close_fp32, col_shards, np64, qkv_shards, unshard_cols,
                     unshard_qkv)
from tensor_transformer_layer_03_b300 import inputs as I

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# (d_model, n_heads, d_ffn, tp, M): ragged M, several tiles, degrees 1..8
SHAPES = [
    (512, 8, 1536, 4, 200),
    (512, 8, 1536, 1, 130),
    (1024, 8, 2816, 8, 77),
    (256, 4, 1024, 2, 1),
    (4096, 32, 11008, 4, 256),
    # small M: the weight-streaming (decode) kernels
    (4096, 32, 11008, 2, 1),
    (4096, 32, 11008, 8, 8),
    (512, 8, 1536, 4, 5),
    (256, 4, 1056, 2, 3),    # 16-row gate/up blocks (d_ffn/tp = 528)
    # 9..32 rows: the weight stream with 2 or 4 groups of 8 token rows
    (4096, 32, 11008, 2, 16),
    (1024, 8, 2816, 4, 24),
    (512, 8, 1536, 2, 32),
    (256, 4, 1056, 2, 12),
    # one-SM tiles (M <= 128) and the edge of the 256-row SM-pair tiles
    (512, 8, 1536, 2, 128),
    (1024, 8, 2816, 4, 100),
    (1024, 8, 2816, 2, 129),
    (512, 8, 1536, 4, 1000),
]


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _plan(tp_mod, d, H, f, deg, act="swiglu", dtype="bf16"):
    return tp_mod.Plan(d, H, f, deg, act=act, dtype=dtype)


def _packed(tp_mod, plan, shape, dtype, seed):
    w = I.make_weights(shape, dtype, _gen(seed))
    pw, _ = plan.sizes(1, 1)
    packed = torch.empty(pw, dtype=torch.uint8, device=DEV)
    plan.shard_weights({k: v.to(DEV) for k, v in w.items()}, packed)
    return w, packed


def _scratch(plan, M, use):
    """Split-tile scratch for the linears, filled with a nonzero byte pattern:
    the ABI ignores its contents on entry (a splitting launch clears its own
    counters).  None: whole tiles only."""
    n = plan.linear_scratch_bytes(M) if use else 0
    return torch.full((n,), 0xA5, dtype=torch.uint8, device=DEV) if n else None


def _again_equal(call, out, what):
    """A second call on the same (already used) scratch gives the same bits."""
    first = out.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(out, first), f"{what}: second call on the same scratch differs"


def _check(got, ref, dtype, what):
    if dtype == "bf16":
        return assert_close_bf16(got, ref, what)
    return assert_close_fp32(got, ref, what)


@pytest.mark.parametrize("sk", [False, True], ids=["tiles", "split"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d,H,f,deg,M", SHAPES)
def test_column_qkv(tp, d, H, f, deg, M, dtype, sk):
    plan = _plan(tp, d, H, f, deg, dtype=dtype)
    shape = I.BlockShape(d, H, f, "swiglu")
    w, packed = _packed(tp, plan, shape, dtype, 1)
    x = I.make_matrix(M, d, dtype, _gen(2))
    out = torch.empty(deg, M, 3 * d // deg, dtype=I.torch_dtype(dtype), device=DEV)
    scr = _scratch(plan, M, sk)
    xd = x.to(DEV)
    plan.column_linear(tp.TP_QKV, xd, M, packed, out, scratch=scr)
    plan.sync_status()
    if scr is not None:
        _again_equal(lambda: plan.column_linear(tp.TP_QKV, xd, M, packed, out, scratch=scr), out, "QKV")
    ref = qkv_shards(o.linear(x, w["Wq"]), o.linear(x, w["Wk"]), o.linear(x, w["Wv"]), deg, H)
    if dtype == "bf16":
        ref = o.round_bf16(ref)
    _check(out, ref, dtype, "QKV")


@pytest.mark.parametrize("sk", [False, True], ids=["tiles", "split"])
@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d,H,f,deg,M", SHAPES)
def test_column_ffn_up(tp, d, H, f, deg, M, dtype, act, sk):
    plan = _plan(tp, d, H, f, deg, act=act, dtype=dtype)
    shape = I.BlockShape(d, H, f, act)
    w, packed = _packed(tp, plan, shape, dtype, 3)
    h = I.make_matrix(M, d, dtype, _gen(4))
    out = torch.empty(deg, M, f // deg, dtype=I.torch_dtype(dtype), device=DEV)
    scr = _scratch(plan, M, sk)
    hd = h.to(DEV)
    plan.column_linear(tp.TP_FFN_UP, hd, M, packed, out, scratch=scr)
    plan.sync_status()
    if scr is not None:
        _again_equal(lambda: plan.column_linear(tp.TP_FFN_UP, hd, M, packed, out, scratch=scr), out, "FFN-up")
    if act == "swiglu":
        u = o.silu(o.linear(h, w["Wg"])) * o.linear(h, w["Wu"])
    else:
        u = o.gelu_erf(o.linear(h, w["W1"]))
    ref = col_shards(u, deg)
    if dtype == "bf16":
        ref = o.round_bf16(ref)
    _check(out, ref, dtype, f"FFN-up {act}")


@pytest.mark.parametrize("sk", [False, True], ids=["tiles", "split"])
@pytest.mark.parametrize("which", ["attn_out", "ffn_down"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d,H,f,deg,M", SHAPES)
def test_row_reduce(tp, d, H, f, deg, M, dtype, which, sk):
    plan = _plan(tp, d, H, f, deg, dtype=dtype)
    shape = I.BlockShape(d, H, f, "swiglu")
    w, packed = _packed(tp, plan, shape, dtype, 5)
    g = _gen(6)
    ks = d // deg if which == "attn_out" else f // deg
    inp = torch.stack([I.make_matrix(M, ks, dtype, g) for _ in range(deg)])
    if which == "attn_out":
        res = I.make_matrix(M, d, dtype, g)
        W = w["Wo"]
        code = tp.TP_ATTN_OUT
    else:
        res = I.make_matrix(M, d, "fp32", g)
        W = w["Wd"]
        code = tp.TP_FFN_DOWN
    out = torch.empty(M, d, dtype=torch.float32, device=DEV)
    out_act = torch.empty(M, d, dtype=I.torch_dtype(dtype), device=DEV)
    scr = _scratch(plan, M, sk)
    ind, resd = inp.to(DEV), res.to(DEV)
    plan.row_linear_reduce(code, ind, M, packed, resd, out, out_act, scratch=scr)
    plan.sync_status()
    if scr is not None:
        _again_equal(lambda: plan.row_linear_reduce(code, ind, M, packed, resd, out, out_act, scratch=scr), out,
                     "row reduce")
    a_full = unshard_cols(inp)
    ref = np64(res) + o.all_reduce_sum(o.row_parallel_partials(a_full, W, deg))
    # fp32 output: accumulation-order noise only.  fp32 plans: <= 1e-5; bf16
    # plans accumulate in the tensor cores' fp32 over K = tp * k_s terms:
    # bound 1e-4 (sqrt(11008) * 2^-24 * a few, with room)
    fp32_bound = 1e-5 if dtype == "fp32" else 1e-4
    nw = float(np.max(np.abs(np64(out) - ref)) / np.max(np.abs(ref)))
    assert nw <= fp32_bound, nw
    _check(out_act, o.round_bf16(ref) if dtype == "bf16" else ref, dtype, "row act copy")
    # without residual and without the act copy
    plan.row_linear_reduce(code, inp.to(DEV), M, packed, None, out, None, scratch=scr)
    plan.sync_status()
    ref0 = ref - np64(res)
    assert float(np.max(np.abs(np64(out) - ref0)) / np.max(np.abs(ref0))) <= fp32_bound


ATTN_CASES = [
    # (d, H, deg, B, T, causal, q_scale)
    (512, 4, 2, 2, 200, True, 1.0),
    (512, 4, 4, 1, 333, False, 1.0),
    (1024, 8, 8, 2, 129, True, 3.0),
    (256, 4, 1, 1, 1, True, 1.0),
    (256, 8, 2, 3, 64, True, 2.0),   # d_head 32
    (4096, 32, 4, 1, 512, True, 1.0),
    # several 128-key steps with large scores: the running max grows by more
    # than 2^8 between steps, so the output rows are rescaled in flight
    (1024, 8, 2, 1, 700, True, 4.0),
    (512, 8, 4, 2, 300, False, 4.0),   # d_head 64, no mask, ragged tail
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d,H,deg,B,T,causal,qs", ATTN_CASES)
def test_attention_prefill(tp, d, H, deg, B, T, causal, qs, dtype):
    plan = _plan(tp, d, H, 8 * deg, deg, dtype=dtype)
    M = B * T
    g = _gen(7)
    qkv = torch.stack([I.make_matrix(M, 3 * d // deg, "fp32", g) for _ in range(deg)])
    c = d // deg
    qkv[:, :, :c] *= qs
    qkv = qkv.to(I.torch_dtype(dtype))
    out = torch.empty(deg, M, d // deg, dtype=I.torch_dtype(dtype), device=DEV)
    plan.attention_heads(qkv.to(DEV), B, T, causal, None, None, 0, 0, out)
    plan.sync_status()
    q, k, v = unshard_qkv(qkv, deg)
    ref = np.concatenate([o.multi_head_attention(q[b * T:(b + 1) * T], k[b * T:(b + 1) * T], v[b * T:(b + 1) * T],
                                                 H, causal) for b in range(B)], axis=0)
    ref = col_shards(ref, deg)
    if dtype == "bf16":
        ref = o.round_bf16(ref)
    _check(out, ref, dtype, "attention")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d,H,deg,B,T,pos,cap", [
    (512, 4, 2, 2, 1, 100, 128),     # single-token decode (split-KV)
    (4096, 32, 2, 1, 1, 1024, 1025),  # the 7B decode shape
    (512, 4, 4, 3, 1, 0, 8),         # first token
    (512, 8, 2, 1, 1, 9000, 9001),   # more keys than 64 chunks of 128
    (512, 4, 2, 2, 37, 50, 100),     # a chunk of tokens after a prefix
    (1024, 8, 4, 1, 300, 200, 640),  # a longer chunk after a prefix, NaN tail
])
def test_attention_with_cache(tp, d, H, deg, B, T, pos, cap, dtype):
    plan = _plan(tp, d, H, 8 * deg, deg, dtype=dtype)
    dh = d // H
    M = B * T
    g = _gen(8)
    qkv = torch.stack([I.make_matrix(M, 3 * d // deg, dtype, g) for _ in range(deg)])
    kc = torch.randn(B, H, cap, dh, generator=g).to(I.torch_dtype(dtype))
    vc = torch.randn(B, H, cap, dh, generator=g).to(I.torch_dtype(dtype))
    # cache rows past the last key are never read: fill them with NaN
    kc[:, :, pos + T:] = float("nan")
    vc[:, :, pos + T:] = float("nan")
    kc_d, vc_d = kc.to(DEV), vc.to(DEV)
    out = torch.empty(deg, M, d // deg, dtype=I.torch_dtype(dtype), device=DEV)
    nscr = plan.attention_scratch_bytes(B, T, cap)
    scratch = torch.empty(max(nscr, 16), dtype=torch.uint8, device=DEV)
    plan.attention_heads(qkv.to(DEV), B, T, True, kc_d, vc_d, cap, pos, out, scratch)
    plan.sync_status()
    q, k, v = unshard_qkv(qkv, deg)
    refs = []
    for b in range(B):
        kk = np.concatenate([np64(kc[b, :, :pos]).transpose(1, 0, 2).reshape(pos, d), k[b * T:(b + 1) * T]])
        vv = np.concatenate([np64(vc[b, :, :pos]).transpose(1, 0, 2).reshape(pos, d), v[b * T:(b + 1) * T]])
        refs.append(o.multi_head_attention(q[b * T:(b + 1) * T], kk, vv, H, True, q_pos0=pos))
    ref = col_shards(np.concatenate(refs, axis=0), deg)
    if dtype == "bf16":
        ref = o.round_bf16(ref)
    _check(out, ref, dtype, "cached attention")
    # the new tokens' K/V landed in the cache at pos.., the rest is untouched
    kn = np64(kc_d.cpu())
    for b in range(B):
        new = k[b * T:(b + 1) * T].reshape(T, H, dh).transpose(1, 0, 2)
        assert np.array_equal(kn[b, :, pos:pos + T], new)
        assert np.array_equal(kn[b, :, :pos], np64(kc[b, :, :pos]))
        assert np.array_equal(kn[b, :, pos + T:], np64(kc[b, :, pos + T:]), equal_nan=True)


@pytest.mark.parametrize("deg,M", [(4, 2048), (2, 128), (4, 512), (4, 4096)])
def test_linears_split_tiles_7b(tp, deg, M):
    """The four linears of the 7B-shaped block at prompt sizes whose tiles
    do not fill the SMs evenly (the last round's tiles cut into parts,
    checked against the host-side schedule query), compared with the oracle
    on sampled rows (rows are independent)."""
    d, H, f = 4096, 32, 11008
    plan = _plan(tp, d, H, f, deg)
    shape = I.BlockShape(d, H, f, "swiglu")
    w, packed = _packed(tp, plan, shape, "bf16", 7)
    g = _gen(8)
    scr = _scratch(plan, M, True)
    nscr = scr.numel()
    rows = sorted(r for r in set([0, 1, 127, 128, M // 2, M - 2, M - 1] + torch.randint(0, M, (9,), generator=g).tolist())
                  if r < M)
    # column QKV and FFN-up
    x = I.make_matrix(M, d, "bf16", g)
    for which, name in ((tp.TP_QKV, "QKV"), (tp.TP_FFN_UP, "FFN-up")):
        sch = plan.linear_schedule(0, which, M, nscr)
        n_out = 3 * d // deg if which == tp.TP_QKV else f // deg
        out = torch.empty(deg, M, n_out, dtype=torch.bfloat16, device=DEV)
        plan.column_linear(which, x.to(DEV), M, packed, out, scratch=scr)
        plan.sync_status()
        xs = x[rows]
        if which == tp.TP_QKV:
            ref = qkv_shards(o.linear(xs, w["Wq"]), o.linear(xs, w["Wk"]), o.linear(xs, w["Wv"]), deg, H)
        else:
            ref = col_shards(o.silu(o.linear(xs, w["Wg"])) * o.linear(xs, w["Wu"]), deg)
        assert_close_bf16(out[:, rows].cpu(), o.round_bf16(ref),
                          f"{name} M={M} tp{deg} (kernel {sch.kernel}, parts {sch.parts}, whole {sch.whole_tiles})")
    # row-parallel O and FFN-down with residual and act copy
    for which, name, ks, W, res_dtype in ((tp.TP_ATTN_OUT, "O", d // deg, w["Wo"], "bf16"),
                                          (tp.TP_FFN_DOWN, "FFN-down", f // deg, w["Wd"], "fp32")):
        sch = plan.linear_schedule(1, which, M, nscr)
        inp = torch.stack([I.make_matrix(M, ks, "bf16", g) for _ in range(deg)])
        res = I.make_matrix(M, d, res_dtype, g)
        out = torch.empty(M, d, dtype=torch.float32, device=DEV)
        out_act = torch.empty(M, d, dtype=torch.bfloat16, device=DEV)
        plan.row_linear_reduce(which, inp.to(DEV), M, packed, res.to(DEV), out, out_act, scratch=scr)
        plan.sync_status()
        ref = np64(res[rows]) + o.all_reduce_sum(o.row_parallel_partials(unshard_cols(inp[:, rows]), W, deg))
        nw = float(np.max(np.abs(np64(out[rows]) - ref)) / np.max(np.abs(ref)))
        assert nw <= 1e-4, (name, M, deg, nw, sch.parts)
        assert_close_bf16(out_act[rows].cpu(), o.round_bf16(ref), f"{name} act copy M={M} tp{deg}")
    # the 128-token prompt (fewer tiles than SMs) cuts every O tile; the
    # 4096-token prompt runs FFN-down's whole rounds and cuts its last one
    if M == 128:
        s = plan.linear_schedule(1, tp.TP_ATTN_OUT, M, nscr)
        assert s.kernel == 0 and not s.paired and s.parts > 1 and s.whole_tiles == 0
    if M == 4096:
        s = plan.linear_schedule(1, tp.TP_FFN_DOWN, M, nscr)
        assert s.kernel == 0 and s.paired and s.parts > 1 and s.whole_tiles > 0
