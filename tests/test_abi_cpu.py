"""The C-ABI library on the CPU: it loads, exports every declared symbol, and
its host-side plan logic and argument validation behave as documented.
No call here reaches a kernel launch (validation fails first)."""
import ctypes
import json
import os
import re

import pytest

import oracle.tp_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tp():
    import __graft_entry__
    __graft_entry__.build()
    from tensor_transformer_layer_03_b300 import tp as binding
    return binding


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(tp_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(tp):
    names = declared_functions()
    assert "tp_block_forward" in names and "tp_plan_create" in names
    for n in names:
        assert hasattr(tp.lib, n), f"{n} declared in include/ but not exported"
        assert n in tp.EXPORTS, f"{n} has no binding"


def _create(tp, d, H, f, deg, act=1, dtype=0):
    h = ctypes.c_void_p()
    code = tp.tp_plan_create_ex(d, H, f, deg, act, dtype, ctypes.byref(h))
    return code, h


def test_plan_rules_match_golden_and_oracle(tp):
    table = json.load(open(os.path.join(ROOT, "tests", "golden", "plan_rules.json")))
    for c in table["cases"]:
        code, h = _create(tp, c["d_model"], c["n_heads"], c["d_ffn"], c["tp"])
        assert tp.status_name(code) == c["expect"] == o.check_plan(c["d_model"], c["n_heads"], c["d_ffn"], c["tp"]), c
        if code == 0:
            assert h.value
            tp.tp_plan_destroy(h)
        else:
            assert not h.value  # *out left NULL on error


def test_plan_rules_exhaustive_small(tp):
    for d in (8, 16, 24, 48, 64):
        for H in range(0, 9):
            for f in (0, 8, 16, 24, 40, 64):
                for deg in range(-1, 10):
                    code, h = _create(tp, d, H, f, deg)
                    exp = o.check_plan(d, H, f, deg)
                    got = tp.status_name(code)
                    if exp == "OK":
                        # the library additionally needs 8-element rows
                        dh, fl = d // H, f // deg
                        exp = "OK" if (d % 8 == 0 and dh % 8 == 0 and fl % 8 == 0) else "ALIGNMENT"
                    assert got == exp, (d, H, f, deg, got, exp)
                    if h.value:
                        tp.tp_plan_destroy(h)


def test_tp_plan_create_defaults_and_null(tp):
    assert tp.tp_plan_create(4096, 32, 11008, 4, None) == 1  # NULL out -> TP_ERR_NULL_ARG
    h = ctypes.c_void_p()
    assert tp.tp_plan_create(5120, 40, 13824, 3, ctypes.byref(h)) == 4  # HEADS_NOT_DIVISIBLE
    assert tp.tp_plan_create(4096, 32, 11008, 4, ctypes.byref(h)) == 0
    tp.tp_plan_destroy(h)
    assert tp.tp_plan_create_ex(256, 4, 1024, 2, 7, 0, ctypes.byref(h)) == 9  # unknown activation


def test_status_strings(tp):
    for i, n in enumerate(tp.STATUS_NAMES):
        assert tp.tp_status_string(i).decode() == ("TP_OK" if n == "OK" else "TP_ERR_" + n)


def test_sizes(tp):
    for (d, H, f, deg, act, dt) in ((4096, 32, 11008, 4, 1, 0), (256, 4, 1024, 2, 0, 1), (5120, 40, 13824, 8, 1, 0)):
        code, h = _create(tp, d, H, f, deg, act, dt)
        assert code == 0
        pw, ws = ctypes.c_size_t(), ctypes.c_size_t()
        assert tp.tp_plan_sizes(h, 2, 128, ctypes.byref(pw), ctypes.byref(ws)) == 0
        es = 2 if dt == 0 else 4
        n_weights = 4 * d * d + (3 if act == 1 else 2) * d * f
        assert n_weights * es <= pw.value <= n_weights * es + 8 * 4096
        M = 256
        acts = M * (3 * d + d + (f if True else 0)) * es + M * d * (4 + es)
        assert ws.value >= acts
        assert tp.tp_plan_sizes(h, 0, 128, ctypes.byref(pw), None) == 2
        assert tp.tp_plan_sizes(None, 1, 1, None, None) == 1
        sb = ctypes.c_size_t()
        assert tp.tp_attention_scratch_bytes(h, 1, 128, 0, ctypes.byref(sb)) == 0 and sb.value == 0
        assert tp.tp_attention_scratch_bytes(h, 2, 1, 1025, ctypes.byref(sb)) == 0 and sb.value > 0
        tp.tp_plan_destroy(h)


def test_argument_validation_before_launch(tp):
    code, h = _create(tp, 256, 4, 1024, 2)
    assert code == 0
    P = lambda v: ctypes.c_void_p(v)  # fake device addresses: never dereferenced
    good, odd = P(0x10000), P(0x10008)
    # column linear
    CL = tp.tp_column_linear
    assert CL(None, 0, good, 4, good, good, None, 0, None) == 1
    assert CL(h, 0, None, 4, good, good, None, 0, None) == 1
    assert CL(h, 0, good, 0, good, good, None, 0, None) == 2
    assert CL(h, 5, good, 4, good, good, None, 0, None) == 2
    assert CL(h, 0, odd, 4, good, good, None, 0, None) == 7
    assert CL(h, 0, good, 4, good, good, odd, 1 << 20, None) == 7   # misaligned scratch
    # row reduce
    RR = tp.tp_row_linear_reduce
    assert RR(h, 0, good, 4, good, None, None, None, None, 0, None) == 1
    assert RR(h, 3, good, 4, good, None, good, None, None, 0, None) == 2
    assert RR(h, 1, good, 4, good, odd, good, None, None, 0, None) == 7
    assert RR(h, 1, good, 4, good, None, good, None, odd, 1 << 20, None) == 7
    # scratch size query
    sb = ctypes.c_size_t()
    assert tp.tp_linear_scratch_bytes(None, 4, ctypes.byref(sb)) == 1
    assert tp.tp_linear_scratch_bytes(h, 0, ctypes.byref(sb)) == 2
    assert tp.tp_linear_scratch_bytes(h, 4, ctypes.byref(sb)) == 0 and sb.value == 0  # weight-streaming rows
    assert tp.tp_linear_scratch_bytes(h, 512, ctypes.byref(sb)) == 0 and sb.value > 0
    # attention
    A = tp.tp_attention_heads
    assert A(h, good, 1, 4, 1, good, None, 8, 0, good, None, 0, None) == 1      # one-sided cache
    assert A(h, good, 1, 4, 1, None, None, 0, 2, good, None, 0, None) == 2      # pos without cache
    assert A(h, good, 1, 4, 1, good, good, 5, 2, good, None, 0, None) == 2      # 2 + 4 > cap 5
    assert A(h, good, 0, 4, 1, None, None, 0, 0, good, None, 0, None) == 2
    assert A(h, good, 1, 1, 1, good, good, 8, 3, good, None, 0, None) == 1      # decode needs scratch
    assert A(h, good, 1, 1, 1, good, good, 8, 3, good, good, 16, None) == 8     # scratch too small
    assert A(h, odd, 1, 4, 1, None, None, 0, 0, good, None, 0, None) == 7
    # block
    B = tp.tp_block_forward
    assert B(h, good, 1, 4, 1, None, None, 0, 0, good, good, 64, good, None) == 8  # workspace too small
    assert B(h, good, 1, 4, 1, None, None, 0, 0, good, None, 1 << 30, good, None) == 1
    assert B(h, good, 1, 0, 1, None, None, 0, 0, good, good, 1 << 30, good, None) == 2
    # more than 2^31 - 1 token rows is refused even with a workspace that claims to be large enough
    assert B(h, good, 1 << 16, 1 << 16, 1, None, None, 0, 0, good, good, (1 << 64) - 1, good, None) == 2
    assert A(h, good, 1 << 16, 1 << 15, 1, None, None, 0, 0, good, None, 0, None) == 2
    # stack
    S = tp.tp_stack_forward
    arr = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    bad = (ctypes.c_void_p * 2)(0x10000, 0)
    odd2 = (ctypes.c_void_p * 2)(0x10000, 0x20008)
    assert S(h, 0, arr, good, 1, 4, 1, None, None, 0, 0, good, 1 << 30, good, None) == 2
    assert S(h, 2, None, good, 1, 4, 1, None, None, 0, 0, good, 1 << 30, good, None) == 1
    assert S(h, 2, bad, good, 1, 4, 1, None, None, 0, 0, good, 1 << 30, good, None) == 1
    assert S(h, 2, odd2, good, 1, 4, 1, None, None, 0, 0, good, 1 << 30, good, None) == 7
    assert S(h, 2, arr, good, 1, 4, 1, arr, None, 8, 0, good, 1 << 30, good, None) == 1   # one-sided caches
    assert S(h, 2, arr, good, 1, 4, 1, None, None, 0, 0, good, 64, good, None) == 8       # workspace too small
    sb = ctypes.c_size_t()
    assert tp.tp_stack_workspace_bytes(h, 1, 4, ctypes.byref(sb)) == 0
    ws = ctypes.c_size_t()
    assert tp.tp_plan_sizes(h, 1, 4, None, ctypes.byref(ws)) == 0 and sb.value > ws.value
    # shard weights: SwiGLU needs Wup
    assert tp.tp_shard_weights(h, good, good, good, good, good, None, good, good, None) == 1
    tp.tp_plan_destroy(h)
    code, h = _create(tp, 256, 4, 1024, 2, act=0)
    assert tp.tp_shard_weights(h, good, good, good, good, good, good, good, good, None) == 1  # GELU: no Wup
    tp.tp_plan_destroy(h)


def test_unsupported_head_width(tp):
    code, h = _create(tp, 192, 4, 64, 2)  # d_head = 48
    assert code == 0
    good = ctypes.c_void_p(0x10000)
    assert tp.tp_attention_heads(h, good, 1, 4, 1, None, None, 0, 0, good, None, 0, None) == 9
    assert tp.tp_attention_decode_noalloc(h, good, 1, good, good, 8, 3, good, None) == 9
    tp.tp_plan_destroy(h)


def test_noalloc_decode_argument_checks(tp):
    """The entry point without allocation checks its arguments and the size
    of its fixed 8 MiB array before anything else: at 32 heads of 128 a
    batch needs 32 * 64 * 130 * 4 bytes of partials, so 7 rows fit and 8 do
    not.  A call that passes the checks on a machine without a GPU stops at
    the device lookup with TP_ERR_CUDA and launches nothing."""
    code, h = _create(tp, 4096, 32, 11008, 2)
    assert code == 0
    P = lambda v: ctypes.c_void_p(v)  # fake device addresses: never dereferenced
    good, odd = P(0x10000), P(0x10008)
    N = tp.tp_attention_decode_noalloc
    assert N(None, good, 1, good, good, 8, 3, good, None) == 1
    for i in range(4):
        args = [good, good, good, good]
        args[i] = None
        q, k, v, out = args
        assert N(h, q, 1, k, v, 8, 3, out, None) == 1
    assert N(h, good, 0, good, good, 8, 3, good, None) == 2     # batch
    assert N(h, good, 1, good, good, 0, 0, good, None) == 2     # capacity
    assert N(h, good, 1, good, good, 8, -1, good, None) == 2    # position
    assert N(h, good, 1, good, good, 8, 8, good, None) == 2     # pos + 1 > cap
    for i in range(4):
        args = [good, good, good, good]
        args[i] = odd
        q, k, v, out = args
        assert N(h, q, 1, k, v, 8, 3, out, None) == 7
    per_row = 32 * 64 * (128 + 2) * 4
    assert 7 * per_row <= (8 << 20) < 8 * per_row
    assert N(h, good, 8, good, good, 8, 3, good, None) == 8     # does not fit the array
    assert N(h, good, 1 << 20, good, good, 8, 3, good, None) == 8
    try:
        import torch
        gpu = torch.cuda.is_available()
    except Exception:
        gpu = True
    if not gpu:
        assert N(h, good, 7, good, good, 8, 3, good, None) == 10  # fits; no device to look up
    tp.tp_plan_destroy(h)


def _create_llama(tp, d, H, f, deg, eps=1e-5, theta=10000.0):
    h = ctypes.c_void_p()
    code = tp.tp_plan_create_llama(d, H, f, deg, eps, theta, ctypes.byref(h))
    return code, h


def test_llama_plan_rules_and_validation(tp):
    """The pre-norm plan: its own argument rules, the block rules of
    tp_plan_create_ex, the 32-row FFN granule, and the calls it refuses."""
    nan, inf = float("nan"), float("inf")
    for eps, theta in ((0.0, 1e4), (-1e-5, 1e4), (nan, 1e4), (inf, 1e4), (1e-5, -1.0), (1e-5, nan), (1e-5, inf)):
        code, h = _create_llama(tp, 256, 4, 1024, 2, eps, theta)
        assert code == 2 and not h.value, (eps, theta)
    assert tp.tp_plan_create_llama(256, 4, 1024, 2, 1e-5, 1e4, None) == 1
    assert _create_llama(tp, 256, 4, 1024, 3)[0] == 4      # heads not divisible by the degree
    assert _create_llama(tp, 256, 4, 1040, 2)[0] == 9      # d_ffn/tp = 520: no 32-row gate/up blocks
    code, h0 = _create(tp, 256, 4, 1024, 2)
    code, h = _create_llama(tp, 256, 4, 1024, 2, theta=0.0)  # theta 0: RMSNorm without rotation
    assert code == 0 and h.value
    good, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
    # column linears of a pre-norm plan need the norm scales: refused
    assert tp.tp_column_linear(h, 0, good, 4, good, good, None, 0, None) == 9
    assert tp.tp_column_linear(h, 1, good, 512, good, good, None, 0, None) == 9
    SW = tp.tp_shard_weights_llama
    args = [good] * 7
    assert SW(h0, *args, good, good, good, None) == 9      # not a pre-norm plan
    assert SW(h, *args, None, good, good, None) == 1
    assert SW(h, *args, good, None, good, None) == 1
    assert SW(h, *args, odd, good, good, None) == 7
    assert SW(h, good, good, good, good, good, None, good, good, good, good, None) == 1  # SwiGLU needs Wup
    # same packed weights, a workspace with room for the 1/rms rows
    pw0, ws0, pw, ws = (ctypes.c_size_t() for _ in range(4))
    assert tp.tp_plan_sizes(h0, 2, 64, ctypes.byref(pw0), ctypes.byref(ws0)) == 0
    assert tp.tp_plan_sizes(h, 2, 64, ctypes.byref(pw), ctypes.byref(ws)) == 0
    assert pw.value == pw0.value and ws.value >= ws0.value + 2 * 128 * 4
    tp.tp_plan_destroy(h)
    tp.tp_plan_destroy(h0)


def test_whole_block_calls_validate_before_the_first_launch(tp):
    """Errors of later steps (attention head width, cache bounds, operand
    alignment) come back before anything is launched: on this GPU-less host
    a launch attempt would report TP_ERR_CUDA instead."""
    P = ctypes.c_void_p
    good, odd = P(0x10000), P(0x10008)
    B = tp.tp_block_forward
    S = tp.tp_stack_forward
    arr = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    code, h = _create(tp, 192, 4, 64, 2)  # d_head = 48: no attention kernel
    assert code == 0
    assert B(h, good, 1, 4, 1, None, None, 0, 0, good, good, 1 << 30, good, None) == 9
    assert S(h, 2, arr, good, 1, 4, 1, None, None, 0, 0, good, 1 << 30, good, None) == 9
    tp.tp_plan_destroy(h)
    for create in (lambda: _create(tp, 256, 4, 1024, 2), lambda: _create_llama(tp, 256, 4, 1024, 2)):
        code, h = create()
        assert code == 0
        assert B(h, good, 1, 4, 1, good, good, 5, 2, good, good, 1 << 30, good, None) == 2   # 2 + 4 > cap 5
        assert B(h, good, 1, 4, 1, good, None, 8, 0, good, good, 1 << 30, good, None) == 1   # one-sided cache
        assert B(h, good, 1, 4, 1, None, None, 0, 3, good, good, 1 << 30, good, None) == 2   # pos without cache
        assert B(h, odd, 1, 4, 1, None, None, 0, 0, good, good, 1 << 30, good, None) == 7    # x
        assert B(h, good, 1, 4, 1, odd, good, 8, 0, good, good, 1 << 30, good, None) == 7    # k cache
        assert B(h, good, 1, 4, 1, None, None, 0, 0, odd, good, 1 << 30, good, None) == 7    # packed
        assert B(h, good, 1, 4, 1, None, None, 0, 0, good, good, 1 << 30, odd, None) == 7    # out
        assert S(h, 2, arr, good, 1, 4, 1, arr, arr, 5, 2, good, 1 << 30, good, None) == 2   # cache bounds
        tp.tp_plan_destroy(h)


def test_sequence_parallel_argument_validation(tp):
    """The sequence-parallel calls check the slicing before anything is
    enqueued: M divisible by tp, slices of a multiple of 8 rows, a stride of
    at least one slice and a multiple of 8 elements, a bf16 plan."""
    P = lambda v: ctypes.c_void_p(v)  # fake device addresses: never dereferenced
    good, odd = P(0x10000), P(0x10008)
    code, h = _create(tp, 256, 4, 1024, 2)  # bf16 SwiGLU, tp 2
    assert code == 0
    G, RS, BS = tp.tp_column_linear_gather, tp.tp_row_linear_reduce_scatter, tp.tp_block_forward_seq
    d, ms = 256, 16                         # M = 32: two slices of 16 rows
    assert G(None, 0, good, ms * d, 32, good, good, None, 0, None) == 1
    assert G(h, 0, good, ms * d, 31, good, good, None, 0, None) == 2           # M not divisible by tp
    assert G(h, 0, good, ms * d, 20, good, good, None, 0, None) == 7           # 10-row slices
    assert G(h, 0, good, ms * d - 8, 32, good, good, None, 0, None) == 2       # stride below a slice
    assert G(h, 0, good, ms * d + 4, 32, good, good, None, 0, None) == 7       # stride not a multiple of 8
    assert G(h, 0, odd, ms * d, 32, good, good, None, 0, None) == 7
    assert G(h, 2, good, ms * d, 32, good, good, None, 0, None) == 2
    assert RS(h, 0, good, 32, good, None, None, None, ms * d, None, 0, None) == 1
    assert RS(h, 1, good, 31, good, None, good, None, ms * d, None, 0, None) == 2
    assert RS(h, 1, good, 32, good, odd, good, None, ms * d, None, 0, None) == 7
    assert RS(h, 1, good, 32, good, None, good, None, 8, None, 0, None) == 2
    assert BS(h, good, ms * d, 1, 32, 1, None, None, 0, 0, good, good, 64, good, ms * d, None) == 8  # workspace
    assert BS(h, good, ms * d, 1, 31, 1, None, None, 0, 0, good, good, 1 << 30, good, ms * d, None) == 2
    assert BS(h, good, ms * d, 1, 32, 1, None, None, 0, 0, good, good, 1 << 30, good, 8, None) == 2  # y stride
    assert BS(h, None, ms * d, 1, 32, 1, None, None, 0, 0, good, good, 1 << 30, good, ms * d, None) == 1
    tp.tp_plan_destroy(h)
    code, h = _create(tp, 256, 4, 1024, 2, dtype=1)  # fp32 plan: no sequence-parallel kernels
    assert code == 0
    assert G(h, 0, good, ms * d, 32, good, good, None, 0, None) == 9
    tp.tp_plan_destroy(h)
