"""Float64 CPU oracle of the Megatron-style tensor-parallel transformer block.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library and never imports it.

Sources (cited by page title and section):

* [TPT] undercodenews.com/?p=110319 (tensor parallelism in transformers),
  section "the Original": attention and the FFN dominate a transformer;
  Q/K/V come from linear projections and are split into heads that attend
  independently and are concatenated; column-parallel = every shard
  multiplies the full input by its slice of the output features;
  row-parallel = the input's column blocks meet the matching row blocks of
  the weight and the partial products are summed by an all-reduce; Q/K/V
  projections are column-parallel so each shard owns a subset of heads and
  attends locally, the output projection is row-parallel; the FFN's first
  linear is column-parallel and its second row-parallel, with an activation
  in between; the degree can exceed neither the head count nor fail to
  divide it, and the FFN width must divide by it.
* [WIT] "What Is Tensor Parallelism?" (netray.co glossary), section
  "Tensor Parallelism Explained": rows or columns are split across cards,
  partial results are combined with an all-reduce, and the degree must divide
  the architectural dimensions such as the head count.
* [BYTE] "Tensor Parallelism: Splitting One Layer Across GPUs" (byteledger),
  section "Interaction with the rest of serving": the KV cache is split along
  with the heads.
* [SP] the same undercodenews page (?p=110319), section "What Undercode
  Say": sequence parallelism spreads the sequence's tokens across the
  devices, combined with tensor parallelism.
* [DMAP] undercodenews "device-map-vs-tensor-parallelism-exposed", section
  "the Original": a model is a sequence of layers, each consuming the
  previous layer's output; device_map places whole layers on different
  devices, tensor parallelism splits every layer.

Readings where the pages are silent (each is listed with its reason in the
design notes):

* activation: GELU is the exact erf form 0.5*x*(1+erf(x/sqrt 2)); SwiGLU is
  silu(x Wg^T) * (x Wu^T) with silu(x) = x / (1 + exp(-x));
* attention scale 1/sqrt(d_head); causal mask where the workload asks for it;
  the mask is applied before the row max, and a query at absolute position p
  sees keys 0..p;
* residual connections are included (H = X + Attn(X), Y = H + FFN(H)); there
  are no norms, biases, RoPE or dropout;
* Q, K and V are each split by head, so shard s owns heads
  [s*h_l, (s+1)*h_l) of all three;
* the all-reduce sums the partials in shard order s = 0..tp-1;
* ``storage="bf16"`` rounds (round-to-nearest-even) the tensors that the
  bf16 data path stores between steps: Q/K/V, the attention output, the bf16
  operand copy of H and U; H itself is kept in fp32 for the residual;
* in a stack of layers the activation passed from one layer to the next is
  stored in the plan dtype (``act_dtype``), in both storage modes;
* the LLaMA-style variant (``llama_block_forward``; norms and rotary
  position embedding are not on the pages) is pre-norm: H = X +
  Attn(RMSNorm(X; g_attn)), Y = H + FFN(RMSNorm(H; g_ffn)), RMSNorm(x; g) =
  x / sqrt(mean(x^2) + eps) * g; RoPE rotates each head's dimension pairs
  (2i, 2i+1) of Q and K by the angle p * theta^(-2i/d_head) at absolute
  position p (the pairing of the original rotary-embedding formulation);
  the KV cache holds the rotated keys;
* sequence parallelism (``sequence_parallel_block_forward``; [SP] names it
  without its mechanics): the token rows of the flattened batch (row
  b*T + t) are cut into tp contiguous slices of M/tp rows; outside the
  tensor-parallel linears and attention, shard s holds only slice s (the
  residual adds happen per slice); the all-reduce after a row-parallel
  linear becomes a reduce-scatter (shard s receives the shard-order sum of
  the partials' rows of its slice) and the input of a column-parallel
  linear is the all-gather (concatenation in shard order) of the slices.

Arrays may be numpy arrays or torch CPU tensors of any float dtype; every
function returns float64 numpy arrays.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

__all__ = [
    "STATUS_NAMES", "check_plan", "to64", "round_bf16", "round_fp32",
    "linear", "gelu_erf", "silu", "softmax_rows", "attention_head",
    "multi_head_attention", "column_parallel_linear", "row_parallel_partials",
    "all_reduce_sum", "ffn", "block_forward", "sharded_block_forward",
    "stack_forward", "rms_norm", "rope", "fold_gains", "llama_block_forward",
    "reduce_scatter_rows", "all_gather_rows", "sequence_parallel_block_forward",
]

# ----------------------------------------------------------------------------
# Degree rule -- [TPT] "the Original" (degree <= head count, head count and
# FFN width divisible by the degree); [WIT] "Tensor Parallelism Explained".
# ----------------------------------------------------------------------------

STATUS_NAMES = (
    "OK", "NULL_ARG", "INVALID_DIM", "DEGREE_RANGE", "HEADS_NOT_DIVISIBLE",
    "FFN_NOT_DIVISIBLE", "DMODEL_NOT_DIVISIBLE",
)


def check_plan(d_model: int, n_heads: int, d_ffn: int, tp: int) -> str:
    """Which rule a (d_model, n_heads, d_ffn, tp) plan breaks first, or "OK".

    Order: positive dimensions; degree at least one; heads of equal width
    (d_model divisible by n_heads); degree no larger than the head count;
    head count divisible by the degree; FFN width divisible by the degree.
    """
    if d_model <= 0 or n_heads <= 0 or d_ffn <= 0:
        return "INVALID_DIM"
    if tp < 1:
        return "DEGREE_RANGE"
    if d_model % n_heads != 0:
        return "DMODEL_NOT_DIVISIBLE"
    if tp > n_heads:
        return "DEGREE_RANGE"
    if n_heads % tp != 0:
        return "HEADS_NOT_DIVISIBLE"
    if d_ffn % tp != 0:
        return "FFN_NOT_DIVISIBLE"
    return "OK"


# ----------------------------------------------------------------------------
# Conversions
# ----------------------------------------------------------------------------

def to64(a) -> np.ndarray:
    """Any float array (numpy, or a torch CPU tensor incl. bf16) as float64."""
    if hasattr(a, "detach"):  # torch tensor: bf16 -> fp32 is exact
        a = a.detach().to("cpu").float().numpy()
    return np.asarray(a, dtype=np.float64)


def round_fp32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_bf16(a) -> np.ndarray:
    """Round to bfloat16 (round to nearest, ties to even), returned as float64.

    The value is first rounded to fp32 and then to bf16 by keeping the top 16
    bits of the fp32 pattern after adding 0x7FFF plus the kept part's lowest
    bit.  (Rounding twice can differ from one direct rounding only for values
    within 2^-24 relative of a bf16 midpoint.)
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _store(a, storage):
    if storage is None:
        return a
    if storage == "bf16":
        return round_bf16(a)
    if storage == "fp32":
        return round_fp32(a)
    raise ValueError(storage)


# ----------------------------------------------------------------------------
# Building blocks
# ----------------------------------------------------------------------------

def linear(x, W) -> np.ndarray:
    """x [.., in] times the transpose of W [out, in] (no bias)."""
    return to64(x) @ to64(W).T


def gelu_erf(x) -> np.ndarray:
    x = to64(x)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def silu(x) -> np.ndarray:
    x = to64(x)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def softmax_rows(s) -> np.ndarray:
    """Softmax over the last axis after subtracting the row max (-inf = masked)."""
    s = to64(s)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_head(q, k, v, causal: bool, q_pos0: int = 0) -> np.ndarray:
    """softmax(q k^T / sqrt(d_head) + mask) v for one head.

    q [Tq, dh] holds the queries at absolute positions q_pos0 .. q_pos0+Tq-1,
    k and v [Tk, dh] the keys/values at positions 0 .. Tk-1.  With ``causal``
    a query at position p only sees keys at positions <= p.
    """
    q, k, v = to64(q), to64(k), to64(v)
    dh = q.shape[-1]
    s = (q @ k.T) / math.sqrt(dh)
    if causal:
        qpos = q_pos0 + np.arange(q.shape[0])[:, None]
        kpos = np.arange(k.shape[0])[None, :]
        s = np.where(kpos > qpos, -np.inf, s)
    return softmax_rows(s) @ v


def multi_head_attention(q, k, v, n_heads: int, causal: bool, q_pos0: int = 0) -> np.ndarray:
    """[TPT] "the Original": every head attends on its own column block of
    Q/K/V and the heads' outputs are concatenated in head order."""
    q, k, v = to64(q), to64(k), to64(v)
    dh = q.shape[-1] // n_heads
    outs = []
    for j in range(n_heads):
        cols = slice(j * dh, (j + 1) * dh)
        outs.append(attention_head(q[:, cols], k[:, cols], v[:, cols], causal, q_pos0))
    return np.concatenate(outs, axis=-1)


def column_parallel_linear(x, W, tp: int) -> list:
    """[TPT] "the Original": shard s multiplies the full input by its own slice
    of the output features (rows [s*n/tp, (s+1)*n/tp) of W [out, in]).  The
    shards' outputs, concatenated in shard order, are x W^T."""
    W = to64(W)
    n = W.shape[0] // tp
    return [linear(x, W[s * n:(s + 1) * n]) for s in range(tp)]


def row_parallel_partials(x, W, tp: int) -> list:
    """[TPT] "the Original": the input's column block s meets the matching
    block of the weight's input features (W[:, block s]); each shard holds a
    partial product of the full output shape."""
    x, W = to64(x), to64(W)
    k = W.shape[1] // tp
    return [x[..., s * k:(s + 1) * k] @ W[:, s * k:(s + 1) * k].T for s in range(tp)]


def all_reduce_sum(partials) -> np.ndarray:
    """The all-reduce of [TPT]/[WIT]: the elementwise sum of the partials,
    taken in shard order."""
    out = np.zeros_like(partials[0])
    for p in partials:
        out = out + p
    return out


def ffn(h, w: dict, act: str, storage=None) -> np.ndarray:
    """Two linears with an activation between ([TPT] "the Original"); U is the
    stored intermediate."""
    if act == "swiglu":
        u = silu(linear(h, w["Wg"])) * linear(h, w["Wu"])
    elif act == "gelu":
        u = gelu_erf(linear(h, w["W1"]))
    else:
        raise ValueError(act)
    return linear(_store(u, storage), w["Wd"])


# ----------------------------------------------------------------------------
# The whole block
# ----------------------------------------------------------------------------

def block_forward(x, w: dict, n_heads: int, act: str, causal: bool,
                  kcache=None, vcache=None, cache_pos: int = 0, storage=None):
    """Unsharded block: Y = H + FFN(H) with H = X + MHA(X) Wo^T.

    x is [B, T, d].  Without a cache the T tokens attend among themselves.
    With ``kcache``/``vcache`` ([B, H, P, d_head], positions 0..cache_pos-1
    valid) the T tokens sit at positions cache_pos .. cache_pos+T-1, their
    keys/values are appended there and they attend over all cache_pos+T keys
    ([BYTE]: the KV cache holds each head's keys/values).

    Returns (Y [B, T, d], K_new [B, H, T, dh], V_new [B, H, T, dh]).
    """
    x = to64(x)
    B, T, d = x.shape
    dh = d // n_heads
    Y = np.empty((B, T, d))
    Kn = np.empty((B, n_heads, T, dh))
    Vn = np.empty((B, n_heads, T, dh))
    for b in range(B):
        xb = x[b]
        q = _store(linear(xb, w["Wq"]), storage)
        k = _store(linear(xb, w["Wk"]), storage)
        v = _store(linear(xb, w["Wv"]), storage)
        Kn[b] = k.reshape(T, n_heads, dh).transpose(1, 0, 2)
        Vn[b] = v.reshape(T, n_heads, dh).transpose(1, 0, 2)
        if kcache is not None:
            kc = to64(kcache[b])[:, :cache_pos]  # [H, P, dh]
            vc = to64(vcache[b])[:, :cache_pos]
            kfull = np.concatenate([kc.transpose(1, 0, 2).reshape(cache_pos, d), k], axis=0)
            vfull = np.concatenate([vc.transpose(1, 0, 2).reshape(cache_pos, d), v], axis=0)
            a = multi_head_attention(q, kfull, vfull, n_heads, causal, q_pos0=cache_pos)
        else:
            a = multi_head_attention(q, k, v, n_heads, causal)
        a = _store(a, storage)
        h = xb + linear(a, w["Wo"])
        h_res = h if storage is None else round_fp32(h)
        h_op = _store(h, storage)
        Y[b] = h_res + ffn(h_op, w, act, storage)
    return Y, Kn, Vn


def sharded_block_forward(x, w: dict, n_heads: int, act: str, causal: bool, tp: int):
    """The same block, computed shard by shard as [TPT] "the Original" lays it
    out: column-parallel Q/K/V by head, local attention over the shard's own
    heads, row-parallel output projection with an all-reduce, column-parallel
    FFN-up (+activation), row-parallel FFN-down with an all-reduce.

    Returns (Y, per-shard attention outputs, per-shard U).
    """
    x = to64(x)
    B, T, d = x.shape
    dh = d // n_heads
    h_l = n_heads // tp
    Wq, Wk, Wv, Wo, Wd = (to64(w[n]) for n in ("Wq", "Wk", "Wv", "Wo", "Wd"))
    up = {n: to64(w[n]) for n in ("Wg", "Wu", "W1") if n in w}
    f = Wd.shape[1]
    f_l = f // tp
    Y = np.empty((B, T, d))
    A_sh, U_sh = [], []
    for b in range(B):
        xb = x[b]
        partials, a_b = [], []
        for s in range(tp):
            rows = slice(s * h_l * dh, (s + 1) * h_l * dh)
            q_s, k_s, v_s = linear(xb, Wq[rows]), linear(xb, Wk[rows]), linear(xb, Wv[rows])
            a_s = multi_head_attention(q_s, k_s, v_s, h_l, causal)
            a_b.append(a_s)
            partials.append(a_s @ Wo[:, rows].T)
        h = xb + all_reduce_sum(partials)
        partials, u_b = [], []
        for s in range(tp):
            cols = slice(s * f_l, (s + 1) * f_l)
            if act == "swiglu":
                u_s = silu(linear(h, up["Wg"][cols])) * linear(h, up["Wu"][cols])
            else:
                u_s = gelu_erf(linear(h, up["W1"][cols]))
            u_b.append(u_s)
            partials.append(u_s @ Wd[:, cols].T)
        Y[b] = h + all_reduce_sum(partials)
        A_sh.append(a_b)
        U_sh.append(u_b)
    return Y, A_sh, U_sh


def reduce_scatter_rows(partials, tp: int) -> list:
    """[SP] reading: the reduce-scatter of the row-parallel partials ([M, n]
    each, M divisible by tp): shard r receives, for the rows of its slice
    [r*M/tp, (r+1)*M/tp) only, the sum of every shard's partial taken in
    shard order."""
    m = partials[0].shape[0]
    ms = m // tp
    out = []
    for r in range(tp):
        acc = np.zeros_like(to64(partials[0][r * ms:(r + 1) * ms]))
        for p in partials:
            acc = acc + to64(p[r * ms:(r + 1) * ms])
        out.append(acc)
    return out


def all_gather_rows(slices) -> np.ndarray:
    """[SP] reading: every shard's input rows, gathered from the shards'
    slices in shard order."""
    return np.concatenate([to64(s) for s in slices], axis=0)


def sequence_parallel_block_forward(x, w: dict, n_heads: int, act: str, causal: bool, tp: int):
    """The block with sequence parallelism around the tensor-parallel
    regions ([SP] with [TPT] "the Original"): x [B, T, d], B*T divisible by
    tp.  Shard s holds token rows slice s of x, H and Y; each column-parallel
    linear reads the all-gathered rows, each row-parallel linear's partials
    are reduce-scattered to the slices and the residual is added per slice.

    Returns (Y [B, T, d] assembled from the slices, [Y slice per shard],
    [H slice per shard])."""
    x = to64(x)
    B, T, d = x.shape
    M = B * T
    if M % tp:
        raise ValueError("B*T must divide by tp")
    ms = M // tp
    dh = d // n_heads
    h_l = n_heads // tp
    Wq, Wk, Wv, Wo, Wd = (to64(w[n]) for n in ("Wq", "Wk", "Wv", "Wo", "Wd"))
    up = {n: to64(w[n]) for n in ("Wg", "Wu", "W1") if n in w}
    f_l = Wd.shape[1] // tp
    x_sl = [x.reshape(M, d)[r * ms:(r + 1) * ms] for r in range(tp)]
    # attention block: all-gather, column-parallel QKV and per-shard heads
    xg = all_gather_rows(x_sl)
    partials = []
    for s in range(tp):
        rows = slice(s * h_l * dh, (s + 1) * h_l * dh)
        a_s = np.empty((M, h_l * dh))
        for b in range(B):
            xb = xg[b * T:(b + 1) * T]
            a_s[b * T:(b + 1) * T] = multi_head_attention(linear(xb, Wq[rows]), linear(xb, Wk[rows]),
                                                          linear(xb, Wv[rows]), h_l, causal)
        partials.append(a_s @ Wo[:, rows].T)
    h_sl = [x_sl[r] + rs for r, rs in enumerate(reduce_scatter_rows(partials, tp))]
    # FFN block: all-gather, column-parallel up (+activation), row-parallel down
    hg = all_gather_rows(h_sl)
    partials = []
    for s in range(tp):
        cols = slice(s * f_l, (s + 1) * f_l)
        if act == "swiglu":
            u_s = silu(linear(hg, up["Wg"][cols])) * linear(hg, up["Wu"][cols])
        else:
            u_s = gelu_erf(linear(hg, up["W1"][cols]))
        partials.append(u_s @ Wd[:, cols].T)
    y_sl = [h_sl[r] + rs for r, rs in enumerate(reduce_scatter_rows(partials, tp))]
    return all_gather_rows(y_sl).reshape(B, T, d), y_sl, h_sl


def stack_forward(x, layers: list, n_heads: int, act: str, causal: bool, kcaches=None, vcaches=None,
                  cache_pos: int = 0, act_dtype: str = "bf16", storage=None):
    """A stack of blocks ([DMAP]: the layers of a model, each consuming the
    previous one's output), every layer tensor-parallel as in block_forward.

    ``layers`` holds one weight dict per layer; ``kcaches``/``vcaches`` one
    cache per layer (or None).  The activation handed to layer l + 1 is
    layer l's Y stored in ``act_dtype`` ("bf16": rounded to bf16; "fp32":
    rounded to fp32).  Returns (last layer's Y, [K_new per layer],
    [V_new per layer]).
    """
    h = to64(x)
    Ks, Vs = [], []
    for i, w in enumerate(layers):
        kw = {}
        if kcaches is not None:
            kw = dict(kcache=kcaches[i], vcache=vcaches[i], cache_pos=cache_pos)
        y, k, v = block_forward(h, w, n_heads, act, causal, storage=storage, **kw)
        Ks.append(k)
        Vs.append(v)
        if i + 1 < len(layers):
            h = round_bf16(y) if act_dtype == "bf16" else round_fp32(y)
        else:
            h = y
    return h, Ks, Vs


# ----------------------------------------------------------------------------
# LLaMA-style pre-norm block (a reading: norms and RoPE are not on the pages)
# ----------------------------------------------------------------------------

def rms_norm(x, g, eps: float) -> np.ndarray:
    """x / sqrt(mean over the last axis of x^2 + eps) * g."""
    x, g = to64(x), to64(g)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x, positions, n_heads: int, theta: float) -> np.ndarray:
    """Rotary position embedding of x [T, n_heads * d_head]: in every head,
    the pair (2i, 2i+1) of token t is rotated by positions[t] * theta^(-2i/d_head)."""
    x = to64(x).copy()
    T, d = x.shape
    dh = d // n_heads
    i = np.arange(dh // 2)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta ** (-2.0 * i / dh)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    for h in range(n_heads):
        ev = x[:, h * dh:(h + 1) * dh:2].copy()
        od = x[:, h * dh + 1:(h + 1) * dh:2].copy()
        x[:, h * dh:(h + 1) * dh:2] = ev * c - od * s
        x[:, h * dh + 1:(h + 1) * dh:2] = ev * s + od * c
    return x


def fold_gains(w: dict, storage) -> dict:
    """The weights with each norm gain folded into the columns that read the
    normed rows: Wq, Wk, Wv times diag(g_attn) and Wg, Wu times diag(g_ffn),
    each product stored once in ``storage``; the gains become 1.  In exact
    arithmetic RMSNorm(x; g) W^T = (x / rms(x)) (W diag(g))^T, so only the
    storage rounding of the products differs from the unfolded form."""
    w = dict(w)
    ga, gf = to64(w["g_attn"]), to64(w["g_ffn"])
    for k in ("Wq", "Wk", "Wv"):
        w[k] = _store(to64(w[k]) * ga[None, :], storage)
    for k in ("Wg", "Wu"):
        w[k] = _store(to64(w[k]) * gf[None, :], storage)
    w["g_attn"], w["g_ffn"] = np.ones_like(ga), np.ones_like(gf)
    return w


def llama_block_forward(x, w: dict, n_heads: int, causal: bool, eps: float, theta: float,
                        kcache=None, vcache=None, cache_pos: int = 0, storage=None, fold: bool = True):
    """Pre-norm block with RMSNorm (w["g_attn"], w["g_ffn"]) and RoPE (theta
    <= 0: none), SwiGLU FFN, tensor-parallel linears as in block_forward.

    x [B, T, d]; the T tokens sit at positions cache_pos..cache_pos+T-1.  The
    norm's 1/rms is taken from the unrounded input; ``storage="bf16"`` rounds
    the same points as block_forward (the normed operand of the FFN is the
    rounded H times that scale) and, with ``fold`` (the default), stores each
    gain folded into the weight columns that read the normed rows
    (``fold_gains``: W diag(g), rounded once, gain then 1).  ``fold=False``
    keeps the gains apart from the weights in storage mode too.  Returns
    (Y, K_new (rotated), V_new).
    """
    x = to64(x)
    if storage is not None and fold:
        w = fold_gains(w, storage)
    B, T, d = x.shape
    dh = d // n_heads
    Y = np.empty((B, T, d))
    Kn = np.empty((B, n_heads, T, dh))
    Vn = np.empty((B, n_heads, T, dh))
    pos = cache_pos + np.arange(T)
    for b in range(B):
        xb = x[b]
        xn = rms_norm(xb, w["g_attn"], eps)
        q, k, v = linear(xn, w["Wq"]), linear(xn, w["Wk"]), linear(xn, w["Wv"])
        if theta > 0:
            q, k = rope(q, pos, n_heads, theta), rope(k, pos, n_heads, theta)
        q, k, v = _store(q, storage), _store(k, storage), _store(v, storage)
        Kn[b] = k.reshape(T, n_heads, dh).transpose(1, 0, 2)
        Vn[b] = v.reshape(T, n_heads, dh).transpose(1, 0, 2)
        if kcache is not None:
            kc = to64(kcache[b])[:, :cache_pos]
            vc = to64(vcache[b])[:, :cache_pos]
            kfull = np.concatenate([kc.transpose(1, 0, 2).reshape(cache_pos, d), k], axis=0)
            vfull = np.concatenate([vc.transpose(1, 0, 2).reshape(cache_pos, d), v], axis=0)
            a = multi_head_attention(q, kfull, vfull, n_heads, causal, q_pos0=cache_pos)
        else:
            a = multi_head_attention(q, k, v, n_heads, causal)
        h = xb + linear(_store(a, storage), w["Wo"])
        h_res = h if storage is None else round_fp32(h)
        scale = 1.0 / np.sqrt(np.mean(h_res * h_res, axis=-1, keepdims=True) + eps)
        hn = _store(h, storage) * scale * to64(w["g_ffn"])
        Y[b] = h_res + ffn(hn, w, "swiglu", storage)
    return Y, Kn, Vn
