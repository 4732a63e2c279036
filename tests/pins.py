"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError when
the oracle disagrees with
  * brute-force pure-Python loops on tiny inputs,
  * library routines in float64 (torch's scaled_dot_product_attention,
    F.linear, F.gelu, F.silu, the bf16 cast),
  * closed forms (causal first row, equal keys, zero weights, Phi(1), ...),
  * identities the pages fix (column-parallel concat, row-parallel partial
    sums, per-head concat, degree invariance of the whole block),
  * the degree-rule table in ``golden/plan_rules.json``.
``test_oracle_mutations.py`` plants plausible mistakes in the oracle and
checks that at least one pin catches each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _weights(rng, d, f, act, std=0.3):
    w = {n: rng.standard_normal((d, d)) * std for n in ("Wq", "Wk", "Wv", "Wo")}
    if act == "swiglu":
        w["Wg"] = rng.standard_normal((f, d)) * std
        w["Wu"] = rng.standard_normal((f, d)) * std
    else:
        w["W1"] = rng.standard_normal((f, d)) * std
    w["Wd"] = rng.standard_normal((d, f)) * std
    return w


# ----------------------------------------------------------------------------
# brute force (pure Python loops, nothing shared with the oracle)
# ----------------------------------------------------------------------------

def bf_matvec_rows(x, W):
    T, K = len(x), len(x[0])
    return [[sum(x[t][k] * W[o][k] for k in range(K)) for o in range(len(W))] for t in range(T)]


def bf_gelu(v):
    return 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))


def bf_silu(v):
    return v / (1.0 + math.exp(-v))


def bf_block_seq(x, w, H, act, causal, kc=None, vc=None, P=0, rnd=None):
    """One sequence.  x: list of T rows of d floats.  kc/vc: [H][P][dh] lists.
    ``rnd`` (optional) rounds a scalar at the bf16 storage points."""
    r = rnd or (lambda v: v)
    T, d = len(x), len(x[0])
    dh = d // H
    q = [[r(v) for v in row] for row in bf_matvec_rows(x, w["Wq"])]
    k = [[r(v) for v in row] for row in bf_matvec_rows(x, w["Wk"])]
    v_ = [[r(v) for v in row] for row in bf_matvec_rows(x, w["Wv"])]
    # full key/value rows: cache rows first (positions 0..P-1), then new tokens
    keys, vals = [], []
    for p in range(P):
        keys.append([kc[h][p][c] for h in range(H) for c in range(dh)])
        vals.append([vc[h][p][c] for h in range(H) for c in range(dh)])
    keys += k
    vals += v_
    a = [[0.0] * d for _ in range(T)]
    for h in range(H):
        for i in range(T):
            qpos = P + i
            js = [j for j in range(len(keys)) if (not causal or j <= qpos)]
            s = [sum(q[i][h * dh + c] * keys[j][h * dh + c] for c in range(dh)) / math.sqrt(dh) for j in js]
            m = max(s)
            e = [math.exp(t - m) for t in s]
            z = sum(e)
            for c in range(dh):
                a[i][h * dh + c] = sum(e[n] * vals[js[n]][h * dh + c] for n in range(len(js))) / z
    a = [[r(v) for v in row] for row in a]
    o = bf_matvec_rows(a, w["Wo"])
    hres = [[x[t][c] + o[t][c] for c in range(d)] for t in range(T)]
    hop = [[r(v) for v in row] for row in hres]
    if act == "swiglu":
        g = bf_matvec_rows(hop, w["Wg"])
        u_ = bf_matvec_rows(hop, w["Wu"])
        u = [[bf_silu(g[t][n]) * u_[t][n] for n in range(len(g[0]))] for t in range(T)]
    else:
        g = bf_matvec_rows(hop, w["W1"])
        u = [[bf_gelu(g[t][n]) for n in range(len(g[0]))] for t in range(T)]
    u = [[r(v) for v in row] for row in u]
    dn = bf_matvec_rows(u, w["Wd"])
    return [[hres[t][c] + dn[t][c] for c in range(d)] for t in range(T)]


def bf_llama_block_seq(x, w, H, causal, eps, theta, kc=None, vc=None, P=0, rnd=None, r32=None, fold=False):
    """Pre-norm RMSNorm + RoPE block on one sequence with explicit loops:
    every pair (2i, 2i+1) of a head rotated with math.cos / math.sin.

    ``rnd`` (optional) rounds a scalar at the bf16 storage points (rotated
    Q/K, V, attention output, the H operand, U) and ``r32`` the residual H;
    with ``fold`` each gain is multiplied into the weight columns that read
    the normed rows and every product is rounded by ``rnd`` on its own
    (g[c] * W[o][c] element by element), the gains then being 1."""
    T, d = len(x), len(x[0])
    dh = d // H
    r = rnd or (lambda v: v)
    f32 = r32 or (lambda v: v)
    if fold:
        w = dict(w)
        for n, gk in (("Wq", "g_attn"), ("Wk", "g_attn"), ("Wv", "g_attn"), ("Wg", "g_ffn"), ("Wu", "g_ffn")):
            w[n] = [[r(row[c] * w[gk][c]) for c in range(len(row))] for row in w[n]]
        w["g_attn"] = [1.0] * d
        w["g_ffn"] = [1.0] * d

    def norm(rows, g):
        out = []
        for row in rows:
            ms = sum(v * v for v in row) / len(row)
            out.append([row[c] / math.sqrt(ms + eps) * g[c] for c in range(len(row))])
        return out

    def rot(rows):
        if theta <= 0:
            return rows
        out = []
        for t, row in enumerate(rows):
            p = P + t
            r2 = list(row)
            for h in range(H):
                for i in range(dh // 2):
                    a, b = row[h * dh + 2 * i], row[h * dh + 2 * i + 1]
                    ang = p * theta ** (-2.0 * i / dh)
                    r2[h * dh + 2 * i] = a * math.cos(ang) - b * math.sin(ang)
                    r2[h * dh + 2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
            out.append(r2)
        return out

    xn = norm(x, w["g_attn"])
    q = [[r(v) for v in row] for row in rot(bf_matvec_rows(xn, w["Wq"]))]
    k = [[r(v) for v in row] for row in rot(bf_matvec_rows(xn, w["Wk"]))]
    v_ = [[r(v) for v in row] for row in bf_matvec_rows(xn, w["Wv"])]
    keys, vals = [], []
    for p in range(P):
        keys.append([kc[h][p][c] for h in range(H) for c in range(dh)])
        vals.append([vc[h][p][c] for h in range(H) for c in range(dh)])
    keys += k
    vals += v_
    a = [[0.0] * d for _ in range(T)]
    for h in range(H):
        for i in range(T):
            js = [j for j in range(len(keys)) if (not causal or j <= P + i)]
            sc = [sum(q[i][h * dh + c] * keys[j][h * dh + c] for c in range(dh)) / math.sqrt(dh) for j in js]
            m = max(sc)
            e = [math.exp(t - m) for t in sc]
            z = sum(e)
            for c in range(dh):
                a[i][h * dh + c] = sum(e[n] * vals[js[n]][h * dh + c] for n in range(len(js))) / z
    a = [[r(v) for v in row] for row in a]
    o_ = bf_matvec_rows(a, w["Wo"])
    hexact = [[x[t][c] + o_[t][c] for c in range(d)] for t in range(T)]
    hres = [[f32(v) for v in row] for row in hexact]
    # the FFN's norm: 1/rms of the residual H, applied to H's bf16 copy
    hn = []
    for t in range(T):
        ms = sum(v * v for v in hres[t]) / d
        sc = 1.0 / math.sqrt(ms + eps)
        hn.append([r(hexact[t][c]) * sc * w["g_ffn"][c] for c in range(d)])
    g = bf_matvec_rows(hn, w["Wg"])
    u_ = bf_matvec_rows(hn, w["Wu"])
    u = [[r(bf_silu(g[t][n]) * u_[t][n]) for n in range(len(g[0]))] for t in range(T)]
    dn = bf_matvec_rows(u, w["Wd"])
    return [[hres[t][c] + dn[t][c] for c in range(d)] for t in range(T)]


def _tolist(w):
    return {n: a.tolist() for n, a in w.items()}


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_brute_force_block(o):
    for act in ("gelu", "swiglu"):
        for causal in (False, True):
            rng = _rng(1 + causal + 2 * (act == "gelu"))
            B, T, d, H, f = 2, 5, 8, 2, 12
            w = _weights(rng, d, f, act)
            x = rng.standard_normal((B, T, d))
            Y, _, _ = o.block_forward(x, w, H, act, causal)
            wl = _tolist(w)
            for b in range(B):
                ref = np.array(bf_block_seq(x[b].tolist(), wl, H, act, causal))
                assert np.max(np.abs(Y[b] - ref)) < 1e-12, (act, causal)


def pin_brute_force_cached(o):
    """Tokens at positions P.. over a filled cache (decode and chunked prefill)."""
    for T, causal in ((1, True), (3, True), (2, False)):
        rng = _rng(7 + T)
        B, d, H, f, P, cap = 2, 8, 2, 6, 4, 9
        dh = d // H
        w = _weights(rng, d, f, "swiglu")
        x = rng.standard_normal((B, T, d))
        kc = rng.standard_normal((B, H, cap, dh))
        vc = rng.standard_normal((B, H, cap, dh))
        Y, Kn, Vn = o.block_forward(x, w, H, "swiglu", causal, kc, vc, P)
        wl = _tolist(w)
        for b in range(B):
            ref = np.array(bf_block_seq(x[b].tolist(), wl, H, "swiglu", causal,
                                        kc[b].tolist(), vc[b].tolist(), P))
            assert np.max(np.abs(Y[b] - ref)) < 1e-12, (T, causal)
            kref = x[b] @ w["Wk"].T
            assert np.max(np.abs(Kn[b].transpose(1, 0, 2).reshape(T, d) - kref)) < 1e-12


def pin_brute_force_bf16_storage(o):
    """The bf16 storage mode equals brute force with torch's bf16 cast at the
    same points (Q/K/V, attention output, H operand, U)."""
    def rnd(v):
        return float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double())
    for act in ("gelu", "swiglu"):
        rng = _rng(31 + (act == "gelu"))
        B, T, d, H, f = 1, 4, 8, 2, 8
        w = _weights(rng, d, f, act)
        x = rng.standard_normal((B, T, d))
        Y, _, _ = o.block_forward(x, w, H, act, True, storage="bf16")
        ref = np.array(bf_block_seq(x[0].tolist(), _tolist(w), H, act, True, rnd=rnd))
        # H keeps an fp32 copy for the residual: compare at fp32 resolution
        assert np.max(np.abs(Y[0] - ref)) < 1e-5 * max(1.0, np.max(np.abs(ref)))
        Y0, _, _ = o.block_forward(x, w, H, act, True)
        assert np.max(np.abs(Y - Y0)) > 1e-6  # the mode really rounds


def pin_torch_attention(o):
    """Per-head attention equals torch's scaled_dot_product_attention (fp64)."""
    rng = _rng(3)
    for causal in (False, True):
        for T, H, dh in ((33, 4, 16), (70, 2, 64), (1, 3, 8)):
            q, k, v = (rng.standard_normal((T, H * dh)) for _ in range(3))
            out = o.multi_head_attention(q, k, v, H, causal)
            tq, tk, tv = (torch.from_numpy(a.reshape(T, H, dh).transpose(1, 0, 2).copy()) for a in (q, k, v))
            ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
            ref = ref.numpy().transpose(1, 0, 2).reshape(T, H * dh)
            assert np.max(np.abs(out - ref)) < 1e-12, (causal, T, H, dh)


def pin_torch_activations(o):
    x = np.concatenate([np.linspace(-40, 40, 4001), _rng(5).standard_normal(1000) * 3])
    tx = torch.from_numpy(x)
    assert np.max(np.abs(o.gelu_erf(x) - F.gelu(tx, approximate="none").numpy())) < 1e-12
    assert np.max(np.abs(o.silu(x) - F.silu(tx).numpy())) < 1e-12


def pin_torch_linear(o):
    rng = _rng(6)
    x, W = rng.standard_normal((7, 13)), rng.standard_normal((5, 13))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(W)).numpy()
    assert np.max(np.abs(o.linear(x, W) - ref)) < 1e-12


def pin_column_parallel(o):
    """Concatenating the column-parallel shards gives the full product."""
    rng = _rng(8)
    x, W = rng.standard_normal((9, 24)), rng.standard_normal((40, 24))
    full = x @ W.T
    for tp in (1, 2, 4, 8):
        shards = o.column_parallel_linear(x, W, tp)
        assert len(shards) == tp and shards[0].shape == (9, 40 // tp)
        assert np.max(np.abs(np.concatenate(shards, axis=1) - full)) < 1e-12


def pin_row_parallel(o):
    """Summing the row-parallel partials gives the full product."""
    rng = _rng(9)
    x, W = rng.standard_normal((9, 32)), rng.standard_normal((12, 32))
    full = x @ W.T
    for tp in (1, 2, 4, 8):
        parts = o.row_parallel_partials(x, W, tp)
        assert len(parts) == tp and parts[0].shape == full.shape
        if tp > 1:
            assert np.max(np.abs(parts[0] - full)) > 1e-3  # a partial is not the whole
        assert np.max(np.abs(o.all_reduce_sum(parts) - full)) < 1e-12


def pin_head_concat(o):
    """Attention over shard-owned head groups, concatenated, is the unsharded MHA."""
    rng = _rng(10)
    T, H, dh = 11, 8, 4
    q, k, v = (rng.standard_normal((T, H * dh)) for _ in range(3))
    full = o.multi_head_attention(q, k, v, H, True)
    for tp in (1, 2, 4, 8):
        h_l = H // tp
        parts = []
        for s in range(tp):
            c = slice(s * h_l * dh, (s + 1) * h_l * dh)
            parts.append(o.multi_head_attention(q[:, c], k[:, c], v[:, c], h_l, True))
        assert np.max(np.abs(np.concatenate(parts, axis=1) - full)) < 1e-12


def pin_degree_invariance(o):
    """The block computed shard by shard equals the unsharded block for every
    degree 1, 2, 4, 8."""
    for act in ("swiglu", "gelu"):
        rng = _rng(11 + (act == "gelu"))
        B, T, d, H, f = 2, 6, 32, 8, 24
        w = _weights(rng, d, f, act)
        x = rng.standard_normal((B, T, d))
        Y, _, _ = o.block_forward(x, w, H, act, True)
        for tp in (1, 2, 4, 8):
            Ys, A, U = o.sharded_block_forward(x, w, H, act, True, tp)
            assert len(A[0]) == tp and A[0][0].shape == (T, d // tp)
            assert len(U[0]) == tp and U[0][0].shape == (T, f // tp)
            assert np.max(np.abs(Ys - Y)) < 1e-11, (act, tp)


def pin_closed_forms_attention(o):
    rng = _rng(12)
    T, dh = 6, 4
    q, k, v = (rng.standard_normal((T, dh)) for _ in range(3))
    # the first query under a causal mask sees only key 0
    assert np.max(np.abs(o.attention_head(q, k, v, True)[0] - v[0])) < 1e-15
    # equal keys: uniform weights, the output is the mean of the visible values
    kk = np.tile(k[:1], (T, 1))
    out = o.attention_head(q, kk, v, False)
    assert np.max(np.abs(out - v.mean(axis=0))) < 1e-12
    outc = o.attention_head(q, kk, v, True)
    run = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(outc - run)) < 1e-12
    # two keys whose scaled scores differ by ln 3: weights 1/4 and 3/4
    q1 = np.array([[2.0 * math.log(3.0), 0.0, 0.0, 0.0]])
    k2 = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    v2 = np.array([[4.0, 0, 0, 0], [0.0, 8.0, 0, 0]])
    assert np.max(np.abs(o.attention_head(q1, k2, v2, False)[0] - np.array([1.0, 6.0, 0, 0]))) < 1e-12
    # a large score difference picks the value of that key
    q3 = np.array([[200.0, 0, 0, 0]])
    assert np.max(np.abs(o.attention_head(q3, k2, v2, False)[0] - v2[1])) < 1e-12
    # softmax: rows sum to one; logs of 1,2,3 give 1/6, 2/6, 3/6
    p = o.softmax_rows(np.log(np.array([[1.0, 2.0, 3.0], [5.0, 5.0, 5.0]])))
    assert np.max(np.abs(p - np.array([[1 / 6, 2 / 6, 3 / 6], [1 / 3] * 3]))) < 1e-15
    p = o.softmax_rows(rng.standard_normal((5, 9)) * 30)
    assert np.max(np.abs(p.sum(axis=1) - 1)) < 1e-14


def pin_closed_forms_activations(o):
    # Phi(1) = 0.841344746068542948... (standard normal CDF), so gelu(1) = Phi(1)
    assert abs(o.gelu_erf(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert abs(o.gelu_erf(np.array([-1.0]))[0] + (1 - 0.8413447460685429)) < 1e-15
    # sigmoid(ln 3) = 3/4
    assert abs(o.silu(np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15
    assert o.gelu_erf(np.array([0.0]))[0] == 0.0 and o.silu(np.array([0.0]))[0] == 0.0
    assert abs(o.gelu_erf(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(o.silu(np.array([-60.0]))[0]) < 1e-20


def pin_closed_forms_block(o):
    """Zero output projections leave Y = X; zero attention weights give the
    running mean of V under a causal mask."""
    rng = _rng(13)
    B, T, d, H, f = 1, 5, 8, 2, 4
    w = _weights(rng, d, f, "swiglu")
    x = rng.standard_normal((B, T, d))
    w0 = dict(w, Wo=np.zeros((d, d)), Wd=np.zeros((d, f)))
    Y, _, _ = o.block_forward(x, w0, H, "swiglu", True)
    assert np.max(np.abs(Y - x)) == 0.0
    # Wq = 0 -> every visible key scores 0 -> attention = running mean of V
    wq0 = dict(w, Wq=np.zeros((d, d)), Wd=np.zeros((d, f)))
    Y, _, _ = o.block_forward(x, wq0, H, "swiglu", True)
    vv = x[0] @ w["Wv"].T
    run = np.cumsum(vv, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(Y[0] - (x[0] + run @ w["Wo"].T))) < 1e-12


def pin_decode_equals_prefill(o):
    """Running the last token over a cache of the earlier tokens' K/V gives the
    prefill's last row, and the appended K/V."""
    rng = _rng(14)
    B, T, d, H, f = 2, 7, 16, 4, 8
    w = _weights(rng, d, f, "swiglu")
    x = rng.standard_normal((B, T, d))
    Y, K, V = o.block_forward(x, w, H, "swiglu", True)
    cap = 10
    kc = np.zeros((B, H, cap, d // H))
    vc = np.zeros((B, H, cap, d // H))
    kc[:, :, :T - 1] = K[:, :, :T - 1]
    vc[:, :, :T - 1] = V[:, :, :T - 1]
    Yd, Kd, Vd = o.block_forward(x[:, T - 1:], w, H, "swiglu", True, kc, vc, T - 1)
    assert np.max(np.abs(Yd[:, 0] - Y[:, T - 1])) < 1e-12
    assert np.max(np.abs(Kd[:, :, 0] - K[:, :, T - 1])) < 1e-12
    assert np.max(np.abs(Vd[:, :, 0] - V[:, :, T - 1])) < 1e-12


def pin_stack_brute_force(o):
    """A 3-layer stack equals brute force applied layer by layer with the
    inter-layer activation rounded to bf16 by torch's cast ([DMAP]: each
    layer consumes the previous one's output)."""
    def rnd_rows(rows):
        return torch.tensor(rows, dtype=torch.float64).to(torch.bfloat16).double().tolist()
    rng = _rng(41)
    B, T, d, H, f, L = 2, 4, 8, 2, 12, 3
    layers = [_weights(rng, d, f, "swiglu") for _ in range(L)]
    x = rng.standard_normal((B, T, d))
    Y, Ks, _ = o.stack_forward(x, layers, H, "swiglu", True)
    for b in range(B):
        h = x[b].tolist()
        for i, w in enumerate(layers):
            h = bf_block_seq(h, _tolist(w), H, "swiglu", True)
            if i + 1 < L:
                h = rnd_rows(h)
        assert np.max(np.abs(Y[b] - np.array(h))) < 1e-12
    assert len(Ks) == L


def pin_stack_closed_forms(o):
    """One layer is the block; layers with zero output projections pass the
    input through (rounded to the inter-layer dtype after every layer but the
    last); a cached 2-layer stack's last decode row equals its prefill."""
    rng = _rng(42)
    B, T, d, H, f = 2, 5, 8, 2, 6
    w = _weights(rng, d, f, "swiglu")
    x = rng.standard_normal((B, T, d))
    Y1, _, _ = o.stack_forward(x, [w], H, "swiglu", True)
    Yb, _, _ = o.block_forward(x, w, H, "swiglu", True)
    assert np.max(np.abs(Y1 - Yb)) == 0.0
    w0 = dict(w, Wo=np.zeros((d, d)), Wd=np.zeros((d, f)))
    Y3, _, _ = o.stack_forward(x, [w0, w0, w0], H, "swiglu", True)
    assert np.max(np.abs(Y3 - o.round_bf16(x))) == 0.0
    Y3f, _, _ = o.stack_forward(x, [w0, w0, w0], H, "swiglu", True, act_dtype="fp32")
    assert np.max(np.abs(Y3f - o.round_fp32(x))) == 0.0
    layers = [_weights(rng, d, f, "swiglu") for _ in range(2)]
    Yp, K, V = o.stack_forward(x, layers, H, "swiglu", True)
    cap, dh = 8, d // H
    kcs = [np.zeros((B, H, cap, dh)) for _ in range(2)]
    vcs = [np.zeros((B, H, cap, dh)) for _ in range(2)]
    for i in range(2):
        kcs[i][:, :, :T - 1] = K[i][:, :, :T - 1]
        vcs[i][:, :, :T - 1] = V[i][:, :, :T - 1]
    Yd, _, _ = o.stack_forward(x[:, T - 1:], layers, H, "swiglu", True, kcs, vcs, T - 1)
    assert np.max(np.abs(Yd[:, 0] - Yp[:, T - 1])) < 1e-12


def _llama_weights(rng, d, f):
    w = _weights(rng, d, f, "swiglu")
    w["g_attn"] = 1.0 + 0.5 * rng.standard_normal(d)
    w["g_ffn"] = 1.0 + 0.5 * rng.standard_normal(d)
    return w


def pin_llama_brute_force(o):
    """The pre-norm RMSNorm + RoPE block against explicit loops, with and
    without a cache (positions offset by the cache length) and without RoPE."""
    for causal, theta, P in ((True, 10000.0, 0), (False, 10000.0, 0), (True, 500.0, 3), (True, 0.0, 0)):
        rng = _rng(51 + P + int(theta) % 7)
        B, T, d, H, f, cap = 2, 4, 8, 2, 6, 7
        w = _llama_weights(rng, d, f)
        x = rng.standard_normal((B, T, d))
        kc = rng.standard_normal((B, H, cap, d // H))
        vc = rng.standard_normal((B, H, cap, d // H))
        kw = dict(kcache=kc, vcache=vc, cache_pos=P) if P else {}
        Y, _, _ = o.llama_block_forward(x, w, H, causal, 1e-5, theta, **kw)
        wl = {n: a.tolist() for n, a in w.items()}
        for b in range(B):
            ref = np.array(bf_llama_block_seq(x[b].tolist(), wl, H, causal, 1e-5, theta,
                                              kc[b].tolist() if P else None, vc[b].tolist() if P else None, P))
            assert np.max(np.abs(Y[b] - ref)) < 1e-11, (causal, theta, P)


def pin_llama_brute_force_bf16_storage(o):
    """The pre-norm block's bf16 storage mode equals explicit loops with
    torch's bf16 cast at the same points: each gain folded into its weight
    columns and every product rounded once, rotated Q/K and V, the attention
    output, H's operand copy and U rounded, H itself kept in fp32.  With
    ``fold=False`` the gains stay apart from the weights."""
    def rnd(v):
        return float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double())

    def r32(v):
        return float(torch.tensor(v, dtype=torch.float64).to(torch.float32).double())
    for causal, theta, P, fold in ((True, 10000.0, 0, True), (True, 500.0, 3, True), (False, 0.0, 0, True),
                                   (True, 10000.0, 2, False)):
        rng = _rng(61 + P + int(theta) % 5 + 7 * fold)
        B, T, d, H, f, cap = 1, 4, 8, 2, 6, 7
        w = _llama_weights(rng, d, f)
        x = rng.standard_normal((B, T, d))
        kc = rng.standard_normal((B, H, cap, d // H))
        vc = rng.standard_normal((B, H, cap, d // H))
        kw = dict(kcache=kc, vcache=vc, cache_pos=P) if P else {}
        Y, _, _ = o.llama_block_forward(x, w, H, causal, 1e-5, theta, storage="bf16", fold=fold, **kw)
        wl = {n: a.tolist() for n, a in w.items()}
        ref = np.array(bf_llama_block_seq(x[0].tolist(), wl, H, causal, 1e-5, theta,
                                          kc[0].tolist() if P else None, vc[0].tolist() if P else None, P,
                                          rnd=rnd, r32=r32, fold=fold))
        # H is an fp32 residual: compare at fp32 resolution
        assert np.max(np.abs(Y[0] - ref)) < 1e-5 * max(1.0, np.max(np.abs(ref))), (causal, theta, P, fold)
        Y0, _, _ = o.llama_block_forward(x, w, H, causal, 1e-5, theta, **kw)
        assert np.max(np.abs(Y - Y0)) > 1e-4  # the mode really rounds
    # folding changes only the rounding: without storage the two forms agree
    rng = _rng(69)
    w = _llama_weights(rng, 8, 6)
    x = rng.standard_normal((1, 3, 8))
    Ya, _, _ = o.llama_block_forward(x, w, 2, True, 1e-5, 10000.0)
    wf = o.fold_gains(w, None)
    assert np.max(np.abs(wf["g_attn"] - 1.0)) == 0.0 and np.max(np.abs(wf["g_ffn"] - 1.0)) == 0.0
    Yb, _, _ = o.llama_block_forward(x, wf, 2, True, 1e-5, 10000.0)
    assert np.max(np.abs(Ya - Yb)) < 1e-12


def pin_reduce_scatter_all_gather(o):
    """The reduce-scatter followed by the all-gather is the all-reduce: the
    slices' sums, gathered in shard order, equal the sum of the whole
    partials, exactly (same terms, same order); each slice holds its own
    rows; gathering returns what was sliced."""
    rng = _rng(71)
    for tp in (1, 2, 4, 8):
        parts = [rng.standard_normal((16, 5)) for _ in range(tp)]
        rs = o.reduce_scatter_rows(parts, tp)
        assert len(rs) == tp and all(r.shape == (16 // tp, 5) for r in rs)
        assert np.array_equal(o.all_gather_rows(rs), o.all_reduce_sum(parts))
        # slice r of shard-order sums, written out with explicit loops
        ms = 16 // tp
        for r in range(tp):
            for i in range(ms):
                for c in range(5):
                    acc = 0.0
                    for p in parts:
                        acc += p[r * ms + i, c]
                    assert abs(rs[r][i, c] - acc) < 1e-12
        x = rng.standard_normal((24, 3))
        assert np.array_equal(o.all_gather_rows([x[i * 24 // tp:(i + 1) * 24 // tp] for i in range(tp)]), x)


def pin_sequence_parallel_block(o):
    """With the tokens sliced across the shards around the tensor-parallel
    regions the block is unchanged: equal to the unsharded block for every
    degree, batch 1 and 2, both activations, with and without the mask; the
    slices are the output's contiguous row blocks."""
    for act in ("swiglu", "gelu"):
        for causal in (True, False):
            rng = _rng(72 + (act == "gelu") + 2 * causal)
            B, T, d, H, f = 2, 8, 16, 8, 24
            w = _weights(rng, d, f, act)
            x = rng.standard_normal((B, T, d))
            Y, _, _ = o.block_forward(x, w, H, act, causal)
            for tp in (1, 2, 4, 8):
                Ys, ysl, hsl = o.sequence_parallel_block_forward(x, w, H, act, causal, tp)
                assert np.max(np.abs(Ys - Y)) < 1e-11, (act, causal, tp)
                assert len(ysl) == tp and ysl[0].shape == (B * T // tp, d)
                assert np.max(np.abs(ysl[-1] - Y.reshape(B * T, d)[-(B * T // tp):])) < 1e-11


def pin_round_fp32(o):
    """Round to fp32, nearest even: 1 + 2^-24 is a tie that goes down to 1,
    1 + 3 * 2^-24 goes up to 1 + 2^-22; against torch's float64 -> float32 cast."""
    got = o.round_fp32(np.array([1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, -(1 + 2.0 ** -24), 0.1, 0.0]))
    assert got[0] == 1.0 and got[1] == 1 + 2.0 ** -22 and got[2] == -1.0 and got[4] == 0.0
    assert got[3] != 0.1 and abs(got[3] - 0.1) < 2.0 ** -27
    x = _rng(17).standard_normal(100000) * np.exp(_rng(18).uniform(-30, 30, 100000))
    ref = torch.from_numpy(x).to(torch.float32).double().numpy()
    assert np.array_equal(o.round_fp32(x), ref)


def pin_rope_properties(o):
    """RoPE equals multiplying each pair, read as a complex number, by
    exp(i p theta^(-2i/dh)); it keeps every pair's norm; position 0 is the
    identity; q at m and k at n score the same as q at m+s and k at n+s."""
    rng = _rng(52)
    T, H, dh, theta = 6, 3, 8, 10000.0
    x = rng.standard_normal((T, H * dh))
    pos = np.array([0, 1, 5, 17, 100, 2047])
    r = o.rope(x, pos, H, theta)
    z = x.reshape(T, H, dh // 2, 2)
    zc = z[..., 0] + 1j * z[..., 1]
    rot = np.exp(1j * pos[:, None, None] * theta ** (-2.0 * np.arange(dh // 2) / dh)[None, None, :])
    ref = zc * rot
    got = r.reshape(T, H, dh // 2, 2)
    assert np.max(np.abs(got[..., 0] - ref.real)) < 1e-12 and np.max(np.abs(got[..., 1] - ref.imag)) < 1e-12
    assert np.max(np.abs(np.abs(got[..., 0] + 1j * got[..., 1]) - np.abs(zc))) < 1e-12
    assert np.max(np.abs(r[0] - x[0])) == 0.0
    q, k = rng.standard_normal((1, dh)), rng.standard_normal((1, dh))
    for m, n, sh in ((3, 1, 7), (10, 10, 100), (0, 5, 33)):
        a = o.rope(q, [m], 1, theta) @ o.rope(k, [n], 1, theta).T
        b = o.rope(q, [m + sh], 1, theta) @ o.rope(k, [n + sh], 1, theta).T
        assert abs(float((a - b).item())) < 1e-10


def pin_rms_norm(o):
    """torch's float64 rms_norm; scale invariance; a constant row c maps to
    sign(c) * g (eps = 0)."""
    rng = _rng(53)
    x = rng.standard_normal((5, 16))
    g = rng.standard_normal(16)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (16,), torch.from_numpy(g), eps=1e-6).numpy()
    assert np.max(np.abs(o.rms_norm(x, g, 1e-6) - ref)) < 1e-12
    assert np.max(np.abs(o.rms_norm(3.7 * x, g, 0.0) - o.rms_norm(x, g, 0.0))) < 1e-12
    c = np.full((2, 16), -2.5)
    assert np.max(np.abs(o.rms_norm(c, g, 0.0) - (-g))) < 1e-12


def pin_llama_decode_equals_prefill(o):
    """The last token decoded over the cache of the earlier tokens' rotated
    K/V equals the prefill's last row."""
    rng = _rng(54)
    B, T, d, H, f = 2, 6, 16, 4, 8
    w = _llama_weights(rng, d, f)
    x = rng.standard_normal((B, T, d))
    Y, K, V = o.llama_block_forward(x, w, H, True, 1e-5, 10000.0)
    kc, vc = np.zeros((B, H, 8, d // H)), np.zeros((B, H, 8, d // H))
    kc[:, :, :T - 1], vc[:, :, :T - 1] = K[:, :, :T - 1], V[:, :, :T - 1]
    Yd, Kd, _ = o.llama_block_forward(x[:, T - 1:], w, H, True, 1e-5, 10000.0, kc, vc, T - 1)
    assert np.max(np.abs(Yd[:, 0] - Y[:, T - 1])) < 1e-12
    assert np.max(np.abs(Kd[:, :, 0] - K[:, :, T - 1])) < 1e-12


def pin_round_bf16(o):
    # ties to even at 1: 1 + 2^-8 -> 1, 1 + 3*2^-8 -> 1 + 2^-6
    vals = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0, 0.0, 1e-30])
    exp = np.array([1.0, 1 + 2.0 ** -6, -1.0, 3.0, 0.0, None], dtype=object)
    got = o.round_bf16(vals)
    for g, e in zip(got[:5], exp[:5]):
        assert g == e
    # against torch's fp32 -> bf16 cast (round to nearest even)
    x = (_rng(15).standard_normal(200000) * np.exp(_rng(16).uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_bf16(x.astype(np.float64)), ref)


def pin_plan_rules(o):
    with open(os.path.join(GOLDEN, "plan_rules.json")) as fh:
        table = json.load(fh)
    for c in table["cases"]:
        got = o.check_plan(c["d_model"], c["n_heads"], c["d_ffn"], c["tp"])
        assert got == c["expect"], (c, got)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
