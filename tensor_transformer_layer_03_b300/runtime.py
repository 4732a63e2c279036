"""Device-side driver of the library: torch allocates, ``libtp.so`` computes.

``TPBlock`` holds one plan, the packed weights and a workspace on a CUDA
device and runs the block through the C ABI.  Torch is used only for device
memory, copies and streams.
"""
from __future__ import annotations

import torch

from . import tp as _tp


_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _norm_device(device) -> torch.device:
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    return dev


def check_tensor(t, name: str, dtype: torch.dtype, device: torch.device, shape=None) -> None:
    """Checks a tensor before its address goes to the library, which reads
    raw pointers with the layouts of include/tp.h: on `device`, of `dtype`,
    contiguous, and of `shape` where given (None entries are not checked)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None:
        if t.dim() != len(shape) or any(e is not None and t.shape[i] != e for i, e in enumerate(shape)):
            want = "[" + ", ".join("*" if e is None else str(e) for e in shape) + "]"
            raise ValueError(f"{name}: shape {list(t.shape)}, expected {want}")


def check_caches(k_cache, v_cache, batch: int, n_heads: int, d_head: int, dtype, device, name="cache") -> None:
    """K and V caches: both or neither, [>= batch][n_heads][cap][d_head]."""
    if (k_cache is None) != (v_cache is None):
        raise ValueError(f"k_{name} and v_{name} must be given together")
    if k_cache is None:
        return
    for t, n in ((k_cache, "k_" + name), (v_cache, "v_" + name)):
        check_tensor(t, n, dtype, device, (None, n_heads, None, d_head))
        if t.shape[0] < batch:
            raise ValueError(f"{n}: {t.shape[0]} sequences, the call has {batch}")
    if k_cache.shape != v_cache.shape:
        raise ValueError(f"k_{name} {list(k_cache.shape)} and v_{name} {list(v_cache.shape)} differ")


def _dev_bytes(nbytes: int, device) -> torch.Tensor:
    # 16-byte aligned by the caching allocator (512-byte granularity); the
    # library ignores a workspace's contents on entry
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


class TPBlock:
    """One tensor-parallel block with its weights resident on ``device``.

    rms_eps given: the pre-norm variant (RMSNorm with the gains
    weights["g_attn"], weights["g_ffn"], rotary embedding with rope_theta)."""

    def __init__(self, shape, tp_degree: int, dtype: str, weights: dict, device="cuda",
                 max_batch: int = 1, max_seq: int = 1, stream=None, rms_eps=None, rope_theta: float = 0.0):
        self.shape, self.tp, self.dtype, self.device = shape, tp_degree, dtype, _norm_device(device)
        self.plan = _tp.Plan(shape.d_model, shape.n_heads, shape.d_ffn, tp_degree, act=shape.act, dtype=dtype,
                             rms_eps=rms_eps, rope_theta=rope_theta)
        packed_bytes, _ = self.plan.sizes(1, 1)
        self.packed = _dev_bytes(packed_bytes, self.device)
        dev_w = {k: v.to(self.device, non_blocking=False).contiguous() for k, v in weights.items()}
        self.plan.shard_weights(dev_w, self.packed, stream)
        torch.cuda.synchronize(self.device)
        del dev_w
        self.workspace = None
        self.reserve(max_batch, max_seq)

    def reserve(self, batch: int, seq: int):
        _, ws = self.plan.sizes(batch, seq)
        if self.workspace is None or self.workspace.numel() < ws:
            self.workspace = _dev_bytes(ws, self.device)

    def forward(self, x: torch.Tensor, causal: bool, out: torch.Tensor | None = None, k_cache=None, v_cache=None,
                cache_pos: int = 0, stream=None) -> torch.Tensor:
        """x: device [B, T, d] in the plan dtype.  Returns Y fp32 [B, T, d]."""
        dt = _TORCH_DTYPE[self.dtype]
        check_tensor(x, "x", dt, self.device, (None, None, self.shape.d_model))
        B, T, d = x.shape
        check_caches(k_cache, v_cache, B, self.shape.n_heads, self.plan.d_head, dt, self.device)
        self.reserve(B, T)
        if out is None:
            out = torch.empty(B, T, d, dtype=torch.float32, device=self.device)
        check_tensor(out, "out", torch.float32, self.device, (B, T, d))
        cap = 0 if k_cache is None else k_cache.shape[2]
        self.plan.block_forward(x, B, T, causal, self.packed, self.workspace, out, k_cache, v_cache, cap, cache_pos,
                                stream)
        return out


    def forward_seq(self, x_slices: torch.Tensor, batch: int, seq: int, causal: bool, out_slices=None, k_cache=None,
                    v_cache=None, cache_pos: int = 0, stream=None) -> torch.Tensor:
        """Sequence-parallel layout: x_slices device [tp][cap][d] in the plan
        dtype, slice s holding token rows s*M/tp .. (s+1)*M/tp - 1 of the
        batch (M = batch * seq) in its first M/tp rows.  Returns Y fp32
        [tp][cap][d] in the same layout (tp_block_forward_seq)."""
        dt = _TORCH_DTYPE[self.dtype]
        check_tensor(x_slices, "x_slices", dt, self.device, (self.tp, None, self.shape.d_model))
        tp, cap, d = x_slices.shape
        check_caches(k_cache, v_cache, batch, self.shape.n_heads, self.plan.d_head, dt, self.device)
        self.reserve(batch, seq)
        if out_slices is None:
            out_slices = torch.empty(tp, cap, d, dtype=torch.float32, device=self.device)
        check_tensor(out_slices, "out_slices", torch.float32, self.device, (tp, None, d))
        kcap = 0 if k_cache is None else k_cache.shape[2]
        self.plan.block_forward_seq(x_slices, cap * d, batch, seq, causal, self.packed, self.workspace, out_slices,
                                    out_slices.shape[1] * d, k_cache, v_cache, kcap, cache_pos, stream)
        return out_slices


class TPStack:
    """n_layers blocks of one shape, each with its own weights on ``device``,
    run through tp_stack_forward (the plan-dtype activation of layer l is the
    input of layer l + 1)."""

    def __init__(self, shape, tp_degree: int, dtype: str, layer_weights: list, device="cuda",
                 max_batch: int = 1, max_seq: int = 1, rms_eps=None, rope_theta: float = 0.0):
        self.blocks = [TPBlock(shape, tp_degree, dtype, w, device=device, max_batch=1, max_seq=1, rms_eps=rms_eps,
                               rope_theta=rope_theta)
                       for w in layer_weights]
        self.plan = self.blocks[0].plan
        self.device = self.blocks[0].device
        self.shape, self.dtype = shape, dtype
        self.workspace = None
        self.reserve(max_batch, max_seq)

    def reserve(self, batch: int, seq: int):
        ws = self.plan.stack_workspace_bytes(batch, seq)
        if self.workspace is None or self.workspace.numel() < ws:
            self.workspace = _dev_bytes(ws, self.device)

    def forward(self, x: torch.Tensor, causal: bool, out: torch.Tensor | None = None, k_caches=None, v_caches=None,
                cache_pos: int = 0, stream=None) -> torch.Tensor:
        """x: device [B, T, d] in the plan dtype.  Returns the last layer's Y
        fp32 [B, T, d].  k_caches / v_caches: one cache per layer, or None."""
        dt = _TORCH_DTYPE[self.dtype]
        check_tensor(x, "x", dt, self.device, (None, None, self.shape.d_model))
        B, T, d = x.shape
        if (k_caches is None) != (v_caches is None):
            raise ValueError("k_caches and v_caches must be given together")
        if k_caches is not None:
            if len(k_caches) != len(self.blocks) or len(v_caches) != len(self.blocks):
                raise ValueError(f"one K and one V cache per layer ({len(self.blocks)} layers)")
            for i, (kc, vc) in enumerate(zip(k_caches, v_caches)):
                check_caches(kc, vc, B, self.shape.n_heads, self.plan.d_head, dt, self.device, f"caches[{i}]")
                if kc.shape != k_caches[0].shape:
                    raise ValueError("every layer's cache must have the shape of layer 0's")
        self.reserve(B, T)
        if out is None:
            out = torch.empty(B, T, d, dtype=torch.float32, device=self.device)
        check_tensor(out, "out", torch.float32, self.device, (B, T, d))
        cap = 0 if k_caches is None else k_caches[0].shape[2]
        self.plan.stack_forward([b.packed for b in self.blocks], x, B, T, causal, self.workspace, out, k_caches,
                                v_caches, cap, cache_pos, stream)
        return out
