"""Plants plausible mistakes in the CPU oracle (on the CPU, through
monkeypatch) and checks that the pins catch every one of them."""
import math

import numpy as np
import pytest

import oracle.tp_oracle as o
from pins import ALL_PINS

real = {n: getattr(o, n) for n in ("attention_head", "linear", "silu", "gelu_erf", "all_reduce_sum",
                                   "block_forward", "round_bf16", "check_plan", "multi_head_attention",
                                   "softmax_rows", "row_parallel_partials", "column_parallel_linear",
                                   "sharded_block_forward", "stack_forward", "rope", "rms_norm", "fold_gains",
                                   "reduce_scatter_rows", "all_gather_rows")}


def _att_scale_dh(q, k, v, causal, q_pos0=0):
    q, k, v = o.to64(q), o.to64(k), o.to64(v)
    return real["attention_head"](q / math.sqrt(q.shape[-1]), k, v, causal, q_pos0)  # 1/d instead of 1/sqrt(d)


def _att_mask_shift(q, k, v, causal, q_pos0=0):
    return real["attention_head"](q, k, v, causal, q_pos0 - 1 if causal else q_pos0)


def _att_no_mask(q, k, v, causal, q_pos0=0):
    return real["attention_head"](q, k, v, False, q_pos0)


def _lt(x, W):
    W = o.to64(W)
    x = o.to64(x)
    if W.shape[0] == W.shape[1]:
        return x @ W  # a square weight used untransposed
    return x @ W.T


def _silu_sign(x):
    x = o.to64(x)
    return x / (1.0 + np.exp(x))


def _gelu_tanh(x):
    x = o.to64(x)
    return 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))


def _reduce_drop_last(parts):
    return real["all_reduce_sum"](parts[:-1]) if len(parts) > 1 else parts[0]


def _block_no_residual(x, w, H, act, causal, *a, **kw):
    Y, K, V = real["block_forward"](x, w, H, act, causal, *a, **kw)
    return Y - o.to64(x), K, V


def _round_truncate(a):
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32) & np.uint32(0xFFFF0000)
    return u.view(np.float32).astype(np.float64)


def _plan_no_ffn(d, H, f, tp):
    r = real["check_plan"](d, H, f, tp)
    return "OK" if r == "FFN_NOT_DIVISIBLE" else r


def _plan_le(d, H, f, tp):
    r = real["check_plan"](d, H, f, tp)
    return "OK" if (r == "DEGREE_RANGE" and tp >= 1) else r


def _mha_wrong_head_cols(q, k, v, n_heads, causal, q_pos0=0):
    # heads taken as interleaved columns instead of contiguous blocks
    q, k, v = o.to64(q), o.to64(k), o.to64(v)
    outs = []
    for j in range(n_heads):
        c = slice(j, None, n_heads)
        outs.append(real["attention_head"](q[:, c], k[:, c], v[:, c], causal, q_pos0))
    return np.concatenate(outs, axis=-1)


def _softmax_no_max(s):
    s = o.to64(s)
    e = np.exp(np.where(np.isinf(s), -np.inf, s))
    return e / np.sum(e, axis=-1, keepdims=True) * (1 + 1e-9)


def _row_wrong_block(x, W, tp):
    x, W = o.to64(x), o.to64(W)
    k = W.shape[1] // tp
    return [x[..., s * k:(s + 1) * k] @ W[:, ((s + 1) % tp) * k:((s + 1) % tp + 1) * k].T for s in range(tp)]


def _col_wrong(x, W, tp):
    W = o.to64(W)
    n = W.shape[0] // tp
    return [o.linear(x, W[s::tp][:n]) for s in range(tp)]


def _stack_no_rounding(x, layers, *a, **kw):
    kw["act_dtype"] = "fp64"  # the inter-layer activation never stored in the plan dtype
    return _stack_fp64(x, layers, *a, **kw)


def _stack_fp64(x, layers, n_heads, act, causal, kcaches=None, vcaches=None, cache_pos=0, act_dtype="bf16",
                storage=None):
    h = o.to64(x)
    for i, w in enumerate(layers):
        kw = {} if kcaches is None else dict(kcache=kcaches[i], vcache=vcaches[i], cache_pos=cache_pos)
        h, _, _ = o.block_forward(h, w, n_heads, act, causal, storage=storage, **kw)
    return h, [], []


def _stack_first_weights(x, layers, *a, **kw):
    return real["stack_forward"](x, [layers[0]] * len(layers), *a, **kw)


def _rope_half(x, positions, n_heads, theta):
    # pairs (i, i + dh/2) instead of (2i, 2i+1)
    x = o.to64(x).copy()
    T, d = x.shape
    dh = d // n_heads
    i = np.arange(dh // 2)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta ** (-2.0 * i / dh)[None, :]
    c, s_ = np.cos(ang), np.sin(ang)
    for h in range(n_heads):
        a = x[:, h * dh:h * dh + dh // 2].copy()
        b = x[:, h * dh + dh // 2:(h + 1) * dh].copy()
        x[:, h * dh:h * dh + dh // 2] = a * c - b * s_
        x[:, h * dh + dh // 2:(h + 1) * dh] = a * s_ + b * c
    return x


def _rope_neg(x, positions, n_heads, theta):
    return real["rope"](x, -np.asarray(positions), n_heads, theta)


def _rms_no_eps(x, g, eps):
    return real["rms_norm"](x, g, 0.0)


def _rms_mean_abs(x, g, eps):
    x, g = o.to64(x), o.to64(g)
    return x / (np.mean(np.abs(x), axis=-1, keepdims=True) + eps) * g


def _fold_unrounded(w, storage):
    # the gain folded into the weights, but the product never stored in bf16
    return real["fold_gains"](w, None)


def _fold_round_twice(w, storage):
    # the weights rounded once more before the gain is folded in
    w = dict(w)
    for k in ("Wq", "Wk", "Wv", "Wg", "Wu"):
        w[k] = o.round_bf16(w[k])
    return real["fold_gains"](w, storage)


def _fold_attn_gain_on_ffn(w, storage):
    # the attention norm's gain folded into the FFN's gate/up columns too
    w = dict(w, g_ffn=w["g_attn"])
    return real["fold_gains"](w, storage)


def _rs_shifted(partials, tp):
    # every shard receives its neighbour's slice
    rs = real["reduce_scatter_rows"](partials, tp)
    return rs[1:] + rs[:1]


def _rs_own_partial_only(partials, tp):
    # each shard keeps its own partial's rows instead of the sum
    ms = partials[0].shape[0] // tp
    return [o.to64(partials[r][r * ms:(r + 1) * ms]) for r in range(tp)]


def _gather_reversed(slices):
    return real["all_gather_rows"](list(slices)[::-1])


MUTATIONS = {
    "reduce-scatter hands out the wrong slice": ("reduce_scatter_rows", _rs_shifted),
    "reduce-scatter skips the sum": ("reduce_scatter_rows", _rs_own_partial_only),
    "all-gather in reverse shard order": ("all_gather_rows", _gather_reversed),
    "folded gain not rounded": ("fold_gains", _fold_unrounded),
    "weights rounded before folding": ("fold_gains", _fold_round_twice),
    "attention gain folded into the FFN": ("fold_gains", _fold_attn_gain_on_ffn),
    "rope pairs (i, i + d/2)": ("rope", _rope_half),
    "rope angle sign": ("rope", _rope_neg),
    "rms norm without eps": ("rms_norm", _rms_no_eps),
    "rms norm by mean |x|": ("rms_norm", _rms_mean_abs),
    "stack skips the inter-layer storage rounding": ("stack_forward", _stack_no_rounding),
    "stack reuses the first layer's weights": ("stack_forward", _stack_first_weights),
    "attention scale 1/d": ("attention_head", _att_scale_dh),
    "causal mask off by one": ("attention_head", _att_mask_shift),
    "causal mask dropped": ("attention_head", _att_no_mask),
    "square weight not transposed": ("linear", _lt),
    "silu sign": ("silu", _silu_sign),
    "gelu tanh form": ("gelu_erf", _gelu_tanh),
    "all-reduce drops a partial": ("all_reduce_sum", _reduce_drop_last),
    "residual dropped": ("block_forward", _block_no_residual),
    "bf16 truncation": ("round_bf16", _round_truncate),
    "FFN divisibility unchecked": ("check_plan", _plan_no_ffn),
    "degree range unchecked": ("check_plan", _plan_le),
    "heads as interleaved columns": ("multi_head_attention", _mha_wrong_head_cols),
    "softmax slightly off": ("softmax_rows", _softmax_no_max),
    "row-parallel mismatched blocks": ("row_parallel_partials", _row_wrong_block),
    "column-parallel strided slices": ("column_parallel_linear", _col_wrong),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(o, attr, bad)
    caught = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(o)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
