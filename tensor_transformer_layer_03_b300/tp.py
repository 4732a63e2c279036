"""ctypes binding of ``libtp.so`` (declared in ``include/tp.h``).

Argument marshalling only: every function keeps the C name and signature,
and tensors are passed as raw device pointers (``tensor.data_ptr()``).  All
work runs in the library's CUDA kernels; there is no Python or CPU
fallback -- if the library is missing, importing this module raises.

``Plan`` is a small convenience wrapper that owns a ``tp_plan_t`` and takes
torch tensors; it only converts arguments and checks status codes.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -m tensor_transformer_layer_03_b300.build` "
                      "(or __graft_entry__.build()) first")
lib = ctypes.CDLL(LIB_PATH)

# ---- enums (same values as include/tp.h) ------------------------------------
TP_OK = 0
STATUS_NAMES = ("OK", "NULL_ARG", "INVALID_DIM", "DEGREE_RANGE", "HEADS_NOT_DIVISIBLE", "FFN_NOT_DIVISIBLE",
                "DMODEL_NOT_DIVISIBLE", "ALIGNMENT", "WORKSPACE_TOO_SMALL", "UNSUPPORTED", "CUDA",
                "DEVICE_TIMEOUT")
TP_ACT_GELU, TP_ACT_SWIGLU = 0, 1
TP_BF16, TP_FP32 = 0, 1
TP_QKV, TP_FFN_UP = 0, 1
TP_ATTN_OUT, TP_FFN_DOWN = 0, 1

_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_plan_p = ctypes.POINTER(ctypes.c_void_p)

EXPORTS = {
    "tp_status_string": (ctypes.c_char_p, [_i]),
    "tp_last_cuda_error": (ctypes.c_char_p, []),
    "tp_plan_create": (_i, [_i, _i, _i, _i, _plan_p]),
    "tp_plan_create_ex": (_i, [_i, _i, _i, _i, _i, _i, _plan_p]),
    "tp_plan_create_llama": (_i, [_i, _i, _i, _i, ctypes.c_float, ctypes.c_float, _plan_p]),
    "tp_plan_destroy": (None, [_p]),
    "tp_plan_sizes": (_i, [_p, _i, _i, ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
    "tp_attention_scratch_bytes": (_i, [_p, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tp_shard_weights": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p]),
    "tp_shard_weights_llama": (_i, [_p] * 12),
    "tp_linear_scratch_bytes": (_i, [_p, _i, ctypes.POINTER(_sz)]),
    "tp_column_linear": (_i, [_p, _i, _p, _i, _p, _p, _p, _sz, _p]),
    "tp_row_linear_reduce": (_i, [_p, _i, _p, _i, _p, _p, _p, _p, _p, _sz, _p]),
    "tp_attention_heads": (_i, [_p, _p, _i, _i, _i, _p, _p, _i, _i, _p, _p, _sz, _p]),
    "tp_block_forward": (_i, [_p, _p, _i, _i, _i, _p, _p, _i, _i, _p, _p, _sz, _p, _p]),
    "tp_attention_decode_noalloc": (_i, [_p, _p, _i, _p, _p, _i, _i, _p, _p]),
    "tp_stack_workspace_bytes": (_i, [_p, _i, _i, ctypes.POINTER(_sz)]),
    "tp_stack_forward": (_i, [_p, _i, ctypes.POINTER(_p), _p, _i, _i, _i, ctypes.POINTER(_p), ctypes.POINTER(_p),
                              _i, _i, _p, _sz, _p, _p]),
    "tp_sync_status": (_i, [_p]),
    "tp_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "tp_column_linear_gather": (_i, [_p, _i, _p, ctypes.c_longlong, _i, _p, _p, _p, _sz, _p]),
    "tp_row_linear_reduce_scatter": (_i, [_p, _i, _p, _i, _p, _p, _p, _p, ctypes.c_longlong, _p, _sz, _p]),
    "tp_block_forward_seq": (_i, [_p, _p, ctypes.c_longlong, _i, _i, _i, _p, _p, _i, _i, _p, _p, _sz, _p,
                                  ctypes.c_longlong, _p]),
    "tp_linear_schedule": (_i, [_p, _i, _i, _i, _sz, _i, _i, _p]),
}


class LinearSchedule(ctypes.Structure):
    """tp_linear_schedule_t."""
    _fields_ = [("kernel", _i), ("paired", _i), ("tiles", _i), ("k_blocks_per_tile", _i), ("whole_tiles", _i),
                ("parts", _i), ("items", _i), ("units", _i), ("scratch_bytes_touched", _sz)]
for _name, (_res, _args) in EXPORTS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args
    globals()[_name] = _f


class TPError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        self.name = STATUS_NAMES[code] if 0 <= code < len(STATUS_NAMES) else f"UNKNOWN({code})"
        msg = f"{where}: TP_ERR_{self.name}" if code else where
        if self.name == "CUDA":
            msg += f" ({tp_last_cuda_error().decode()})"
        super().__init__(msg)


def check(code: int, where: str = "") -> None:
    if code != TP_OK:
        raise TPError(code, where)


def status_name(code: int) -> str:
    return STATUS_NAMES[code]


def _ptr(t):
    """Device address of a CUDA tensor (None for NULL).  Every buffer
    argument of the library is device memory, so a host tensor is refused
    here: a kernel given its address would fault."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Owns a tp_plan_t.  Methods take torch tensors (device pointers)."""

    def __init__(self, d_model, n_heads, d_ffn, tp_degree, act="swiglu", dtype="bf16", rms_eps=None,
                 rope_theta=0.0):
        """rms_eps given: the pre-norm (RMSNorm + RoPE) variant, which is
        SwiGLU and bf16 only (tp_plan_create_llama)."""
        h = ctypes.c_void_p()
        self.llama = rms_eps is not None
        if self.llama:
            if act != "swiglu" or dtype != "bf16":
                raise ValueError("the pre-norm block is SwiGLU and bf16")
            code = tp_plan_create_llama(d_model, n_heads, d_ffn, tp_degree, float(rms_eps), float(rope_theta),
                                        ctypes.byref(h))
            check(code, "tp_plan_create_llama")
        else:
            code = tp_plan_create_ex(d_model, n_heads, d_ffn, tp_degree,
                                     TP_ACT_SWIGLU if act == "swiglu" else TP_ACT_GELU,
                                     TP_BF16 if dtype == "bf16" else TP_FP32, ctypes.byref(h))
            check(code, "tp_plan_create_ex")
        self.handle = h
        self.d_model, self.n_heads, self.d_ffn, self.tp = d_model, n_heads, d_ffn, tp_degree
        self.d_head = d_model // n_heads
        self.h_l, self.f_l = n_heads // tp_degree, d_ffn // tp_degree
        self.act, self.dtype = act, dtype

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            tp_plan_destroy(h)
            self.handle = None

    def sizes(self, batch, seq):
        pw, ws = _sz(), _sz()
        check(tp_plan_sizes(self.handle, batch, seq, ctypes.byref(pw), ctypes.byref(ws)), "tp_plan_sizes")
        return pw.value, ws.value

    def attention_scratch_bytes(self, batch, seq_q, cache_cap):
        b = _sz()
        check(tp_attention_scratch_bytes(self.handle, batch, seq_q, cache_cap, ctypes.byref(b)),
              "tp_attention_scratch_bytes")
        return b.value

    def shard_weights(self, w: dict, packed, stream=None):
        up = w.get("Wu")
        first = w["Wg"] if up is not None else w["W1"]
        if self.llama:
            check(tp_shard_weights_llama(self.handle, _ptr(w["Wq"]), _ptr(w["Wk"]), _ptr(w["Wv"]), _ptr(w["Wo"]),
                                         _ptr(first), _ptr(up), _ptr(w["Wd"]), _ptr(w["g_attn"]), _ptr(w["g_ffn"]),
                                         _ptr(packed), _stream(stream)), "tp_shard_weights_llama")
            return
        check(tp_shard_weights(self.handle, _ptr(w["Wq"]), _ptr(w["Wk"]), _ptr(w["Wv"]), _ptr(w["Wo"]),
                               _ptr(first), _ptr(up), _ptr(w["Wd"]), _ptr(packed), _stream(stream)),
              "tp_shard_weights")

    def linear_schedule(self, row, which, M, scratch_bytes, sms=148, pair_slots=74):
        """Host-only: how the linear would run (tp_linear_schedule)."""
        out = LinearSchedule()
        check(tp_linear_schedule(self.handle, int(row), which, M, scratch_bytes, sms, pair_slots,
                                 ctypes.cast(ctypes.byref(out), ctypes.c_void_p)), "tp_linear_schedule")
        return out

    def linear_scratch_bytes(self, M):
        b = _sz()
        check(tp_linear_scratch_bytes(self.handle, M, ctypes.byref(b)), "tp_linear_scratch_bytes")
        return b.value

    def column_linear(self, which, x, M, packed, out, stream=None, scratch=None):
        nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
        check(tp_column_linear(self.handle, which, _ptr(x), M, _ptr(packed), _ptr(out), _ptr(scratch), nbytes,
                               _stream(stream)), "tp_column_linear")

    def column_linear_gather(self, which, x_slices, slice_stride, M, packed, out, stream=None, scratch=None):
        """x_slices: a tensor whose storage holds tp slices of M / tp rows,
        slice_stride elements apart (tp_column_linear_gather)."""
        nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
        check(tp_column_linear_gather(self.handle, which, _ptr(x_slices), slice_stride, M, _ptr(packed), _ptr(out),
                                      _ptr(scratch), nbytes, _stream(stream)), "tp_column_linear_gather")

    def row_linear_reduce_scatter(self, which, inp, M, packed, residual, out_f32, out_act, slice_stride, stream=None,
                                  scratch=None):
        nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
        check(tp_row_linear_reduce_scatter(self.handle, which, _ptr(inp), M, _ptr(packed), _ptr(residual),
                                           _ptr(out_f32), _ptr(out_act), slice_stride, _ptr(scratch), nbytes,
                                           _stream(stream)), "tp_row_linear_reduce_scatter")

    def block_forward_seq(self, x_slices, x_stride, batch, seq, causal, packed, workspace, out_slices, y_stride,
                          k_cache=None, v_cache=None, cache_cap=0, cache_pos=0, stream=None):
        nbytes = workspace.numel() * workspace.element_size()
        check(tp_block_forward_seq(self.handle, _ptr(x_slices), x_stride, batch, seq, 1 if causal else 0,
                                   _ptr(k_cache), _ptr(v_cache), cache_cap, cache_pos, _ptr(packed), _ptr(workspace),
                                   nbytes, _ptr(out_slices), y_stride, _stream(stream)), "tp_block_forward_seq")

    def row_linear_reduce(self, which, inp, M, packed, residual, out_f32, out_act=None, stream=None, scratch=None):
        nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
        check(tp_row_linear_reduce(self.handle, which, _ptr(inp), M, _ptr(packed), _ptr(residual),
                                   _ptr(out_f32), _ptr(out_act), _ptr(scratch), nbytes, _stream(stream)),
              "tp_row_linear_reduce")

    def attention_heads(self, qkv, batch, seq_q, causal, k_cache, v_cache, cache_cap, cache_pos, out,
                        scratch=None, stream=None):
        nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
        check(tp_attention_heads(self.handle, _ptr(qkv), batch, seq_q, int(causal), _ptr(k_cache), _ptr(v_cache),
                                 cache_cap, cache_pos, _ptr(out), _ptr(scratch), nbytes, _stream(stream)),
              "tp_attention_heads")

    def block_forward(self, x, batch, seq, causal, packed, workspace, out_f32, k_cache=None, v_cache=None,
                      cache_cap=0, cache_pos=0, stream=None):
        nbytes = workspace.numel() * workspace.element_size()
        check(tp_block_forward(self.handle, _ptr(x), batch, seq, int(causal), _ptr(k_cache), _ptr(v_cache),
                               cache_cap, cache_pos, _ptr(packed), _ptr(workspace), nbytes, _ptr(out_f32),
                               _stream(stream)), "tp_block_forward")

    def attention_decode_noalloc(self, qkv, batch, k_cache, v_cache, cache_cap, cache_pos, out, stream=None):
        check(tp_attention_decode_noalloc(self.handle, _ptr(qkv), batch, _ptr(k_cache), _ptr(v_cache), cache_cap,
                                          cache_pos, _ptr(out), _stream(stream)), "tp_attention_decode_noalloc")

    def stack_workspace_bytes(self, batch, seq):
        b = _sz()
        check(tp_stack_workspace_bytes(self.handle, batch, seq, ctypes.byref(b)), "tp_stack_workspace_bytes")
        return b.value

    def stack_forward(self, packed_layers, x, batch, seq, causal, workspace, out_f32, k_caches=None, v_caches=None,
                      cache_cap=0, cache_pos=0, stream=None):
        n = len(packed_layers)
        arr = lambda ts: (ctypes.c_void_p * n)(*[_ptr(t).value for t in ts]) if ts is not None else None
        nbytes = workspace.numel() * workspace.element_size()
        check(tp_stack_forward(self.handle, n, arr(packed_layers), _ptr(x), batch, seq, int(causal), arr(k_caches),
                               arr(v_caches), cache_cap, cache_pos, _ptr(workspace), nbytes, _ptr(out_f32),
                               _stream(stream)), "tp_stack_forward")

    def sync_status(self, stream=None):
        check(tp_sync_status(_stream(stream)), "tp_sync_status")
