"""GPU parity of the whole block (tp_block_forward) against the float64
oracle, for every degree 1/2/4/8, at the workloads' full sizes.

Bounds (see helpers.py): fp32 path normwise <= 1e-5; bf16 path normwise
<= 2e-2 against the exact oracle and mean abs <= max(1e-3, 1.25 x floor),
floor = mean |oracle(bf16 storage) - oracle(exact)| on the same inputs.
Batches larger than the oracle can redo in seconds are checked on their
first and last sequences (sequences are independent)."""
import numpy as np
import pytest
import torch

import oracle.tp_oracle as o
from helpers import BF16_MEAN_ABS, FLOOR_FACTOR, assert_close_bf16, assert_close_fp32, mean_abs, np64
from tensor_transformer_layer_03_b300 import inputs as I
from tensor_transformer_layer_03_b300.runtime import TPBlock

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

_ORACLE = {}


def _oracle(key, inp, wl, seqs=None, cache=None):
    """(exact Y, bf16-storage Y) for the selected sequences, memoised."""
    k = (key, tuple(seqs) if seqs is not None else None)
    if k not in _ORACLE:
        w = {n: v for n, v in inp.items() if n.startswith("W")}
        x = inp["X"] if seqs is None else inp["X"][list(seqs)]
        kw = {}
        if cache is not None:
            kw = dict(kcache=cache[0], vcache=cache[1], cache_pos=cache[2])
        ex, K, V = o.block_forward(x, w, wl.shape.n_heads, wl.shape.act, wl.causal, **kw)
        st = None
        if wl.dtype == "bf16":
            st, _, _ = o.block_forward(x, w, wl.shape.n_heads, wl.shape.act, wl.causal, storage="bf16", **kw)
        _ORACLE[k] = (ex, st, K, V)
    return _ORACLE[k]


def _check_block(got, ex, st, dtype, what):
    if dtype == "fp32":
        return assert_close_fp32(got, ex, what)
    floor = mean_abs(st, ex)
    return assert_close_bf16(got, ex, what, mean_abs_bound=max(BF16_MEAN_ABS, FLOOR_FACTOR * floor))


def _run(wl, inp, causal=None):
    w = {n: v for n, v in inp.items() if n.startswith("W")}
    blk = TPBlock(wl.shape, wl.tp, wl.dtype, w, device=DEV, max_batch=wl.batch, max_seq=wl.seq)
    y = blk.forward(inp["X"].to(DEV), wl.causal if causal is None else causal)
    blk.plan.sync_status()
    return y.cpu(), blk


def test_tiny_fp32_block(tp):
    wl = I.WORKLOADS["tiny_fp32"]
    inp = I.make_inputs(wl)
    y, _ = _run(wl, inp)
    ex, _, _, _ = _oracle("tiny", inp, wl)
    _check_block(y, ex, None, "fp32", "tiny fp32")


SMALL = I.BlockShape(512, 8, 1536, "swiglu")


@pytest.mark.parametrize("deg", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype,act", [("bf16", "swiglu"), ("bf16", "gelu"), ("fp32", "swiglu")])
def test_small_block_all_degrees(tp, deg, dtype, act):
    wl = I.Workload("small", I.BlockShape(512, 8, 1536, act), tp=deg, batch=2, seq=160, causal=True, dtype=dtype)
    inp = I.make_inputs(wl, seed=3)
    y, _ = _run(wl, inp)
    ex, st, _, _ = _oracle(("small", act, dtype), inp, wl)
    _check_block(y, ex, st, dtype, f"small tp{deg} {dtype} {act}")


def test_degree_invariance_on_gpu(tp):
    """tp=1 and tp=2,4,8 give the same block up to bf16 rounding noise."""
    outs = {}
    for deg in (1, 2, 4, 8):
        wl = I.Workload("inv", SMALL, tp=deg, batch=1, seq=96, causal=True, dtype="bf16")
        outs[deg], _ = _run(wl, I.make_inputs(wl, seed=5))
    for deg in (2, 4, 8):
        d = np64(outs[deg]) - np64(outs[1])
        assert np.max(np.abs(d)) / np.max(np.abs(np64(outs[1]))) <= 2e-2
        assert np.mean(np.abs(d)) <= 2e-3


@pytest.mark.parametrize("deg", [1, 2, 4, 8])
def test_llama7b_block_t256_all_degrees(tp, deg):
    wl = I.WORKLOADS["llama7b_prefill"].with_(tp=deg, seq=256)
    inp = I.make_inputs(wl)
    y, _ = _run(wl, inp)
    ex, st, _, _ = _oracle("7b_t256", inp, wl)
    _check_block(y, ex, st, "bf16", f"7B T256 tp{deg}")


def test_llama7b_prefill_full(tp):
    wl = I.WORKLOADS["llama7b_prefill"]
    inp = I.make_inputs(wl)
    y, _ = _run(wl, inp)
    ex, st, _, _ = _oracle("7b_full", inp, wl)
    _check_block(y, ex, st, "bf16", "7B prefill B1xT2048 tp4")


def test_llama7b_decode_full(tp):
    wl = I.WORKLOADS["llama7b_decode"]
    inp = I.make_inputs(wl)
    w = {n: v for n, v in inp.items() if n.startswith("W")}
    cap = wl.cache_len + 1
    B, H, dh = wl.batch, wl.shape.n_heads, wl.shape.d_head
    kc = torch.zeros(B, H, cap, dh, dtype=torch.bfloat16)
    vc = torch.zeros(B, H, cap, dh, dtype=torch.bfloat16)
    kc[:, :, :wl.cache_len] = inp["Kcache"]
    vc[:, :, :wl.cache_len] = inp["Vcache"]
    kd, vd = kc.to(DEV), vc.to(DEV)
    blk = TPBlock(wl.shape, wl.tp, wl.dtype, w, device=DEV, max_batch=B, max_seq=1)
    y = blk.forward(inp["X"].to(DEV), True, k_cache=kd, v_cache=vd, cache_pos=wl.cache_len)
    blk.plan.sync_status()
    ex, st, K, V = _oracle("7b_decode", inp, wl, cache=(kc, vc, wl.cache_len))
    _check_block(y.cpu(), ex, st, "bf16", "7B decode tp2")
    # appended K/V: the bf16 values the GPU stored vs the oracle's exact ones
    assert_close_bf16(kd[:, :, wl.cache_len].cpu(), o.round_bf16(K[:, :, 0]), "appended K")
    assert_close_bf16(vd[:, :, wl.cache_len].cpu(), o.round_bf16(V[:, :, 0]), "appended V")


@pytest.mark.parametrize("deg", [1, 2, 4, 8])
def test_llama13b_tp_sweep(tp, deg):
    wl = I.WORKLOADS["llama13b_b4t1024"].with_(tp=deg)
    inp = I.make_inputs(wl)
    y, _ = _run(wl, inp)
    ex, st, _, _ = _oracle("13b", inp, wl)
    _check_block(y, ex, st, "bf16", f"13B B4xT1024 tp{deg}")


@pytest.mark.parametrize("B", I.SWEEP_BATCH)
@pytest.mark.parametrize("T", I.SWEEP_SEQ)
def test_llama7b_sweep_sampled(tp, B, T):
    wl = I.WORKLOADS["llama7b_prefill"].with_(batch=B, seq=T)
    inp = I.make_inputs(wl)
    y, _ = _run(wl, inp)
    seqs = sorted({0, B - 1})
    ex, st, _, _ = _oracle(("sweep", B, T), inp, wl, seqs=seqs)
    _check_block(y[seqs], ex, st, "bf16", f"7B sweep B{B} T{T} (sequences {seqs})")


def test_workspace_reused_across_shapes():
    """One workspace serves prompts of different sizes in turn: the linears'
    split-tile counters sit at an offset that moves with the token count, on
    bytes an earlier, larger call used for activations.  Every call must
    still finish (no device timeout) and give the bits of a block whose
    workspace holds an arbitrary byte pattern."""
    shape, deg = I.LLAMA7B, 4
    g = torch.Generator().manual_seed(21)
    w = I.make_weights(shape, "bf16", g)
    blk = TPBlock(shape, deg, "bf16", w, device=DEV)
    fresh = TPBlock(shape, deg, "bf16", w, device=DEV)
    for B, T in ((1, 2048), (4, 128), (1, 512), (2, 64), (1, 2048)):
        x = torch.randn(B, T, shape.d_model, generator=g).to(torch.bfloat16).to(DEV)
        y = blk.forward(x, True)
        blk.plan.sync_status()
        fresh.workspace = None
        fresh.reserve(B, T)
        fresh.workspace.fill_(0xA5)
        y2 = fresh.forward(x, True)
        fresh.plan.sync_status()
        assert torch.equal(y, y2), (B, T)
