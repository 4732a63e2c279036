"""Seeded synthetic inputs for the tensor-parallel transformer block.

This module is shared by the tests (which feed the same tensors to the CPU
oracle and to the CUDA library), by ``bench.py`` and by ``smoke()``.  It holds
none of the block's arithmetic: only the workload shapes, the random draws,
the scaling of those draws and the cast to the storage dtype.

Recipe (the same for every workload):

* one ``torch.Generator`` on the CPU, ``manual_seed(seed)`` (seed 0 unless a
  test says otherwise);
* fp32 ``randn`` draws in this fixed order: Wq, Wk, Wv, Wo, then Wg, Wu
  (SwiGLU) or W1 (GELU), then Wd, then the activations X, then (decode only)
  the K cache and the V cache;
* weight draws are multiplied by 0.02 (weights N(0, 0.02^2)); activations and
  cache entries stay N(0, 1);
* every tensor is then cast to the workload's storage dtype (bf16 or fp32).
  Both sides consume the cast values, so input quantisation is not error.

Weights use the PyTorch ``[out_features, in_features]`` row-major layout:
Wq/Wk/Wv/Wo are [d, d], Wg/Wu/W1 are [f, d], Wd is [d, f].  X is [B, T, d];
the caches are [B, H, cache_len, d_head] with positions 0..cache_len-1 filled.
"""
from __future__ import annotations

import dataclasses

import torch

WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class BlockShape:
    d_model: int
    n_heads: int
    d_ffn: int
    act: str  # "gelu" or "swiglu"

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_heads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: BlockShape
    tp: int
    batch: int
    seq: int
    causal: bool
    dtype: str  # "bf16" or "fp32"
    decode: bool = False
    cache_len: int = 0  # prior positions already in the cache (decode)

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = BlockShape(d_model=256, n_heads=4, d_ffn=1024, act="gelu")
LLAMA7B = BlockShape(d_model=4096, n_heads=32, d_ffn=11008, act="swiglu")
LLAMA13B = BlockShape(d_model=5120, n_heads=40, d_ffn=13824, act="swiglu")

# The five workloads the block is exercised on.  The tiny one has no mask
# (nothing asks for one); the 13B-shaped one is causal like the 7B one.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", TINY, tp=2, batch=1, seq=64, causal=False, dtype="fp32"),
    "llama7b_prefill": Workload("llama7b_prefill", LLAMA7B, tp=4, batch=1, seq=2048, causal=True, dtype="bf16"),
    "llama7b_decode": Workload("llama7b_decode", LLAMA7B, tp=2, batch=1, seq=1, causal=True, dtype="bf16",
                               decode=True, cache_len=1024),
    "llama13b_b4t1024": Workload("llama13b_b4t1024", LLAMA13B, tp=4, batch=4, seq=1024, causal=True, dtype="bf16"),
}
SWEEP_BATCH = (1, 4, 16, 64)
SWEEP_SEQ = (128, 512, 2048)
TP_SWEEP = (1, 2, 4, 8)


def sweep_workloads():
    base = WORKLOADS["llama7b_prefill"]
    return [base.with_(name=f"llama7b_b{b}_t{t}", batch=b, seq=t) for b in SWEEP_BATCH for t in SWEEP_SEQ]


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]


def make_weights(shape: BlockShape, dtype: str, gen: torch.Generator) -> dict:
    d, f = shape.d_model, shape.d_ffn
    dt = torch_dtype(dtype)

    def w(rows, cols):
        return (torch.randn(rows, cols, generator=gen) * WEIGHT_STD).to(dt)

    out = {"Wq": w(d, d), "Wk": w(d, d), "Wv": w(d, d), "Wo": w(d, d)}
    if shape.act == "swiglu":
        out["Wg"] = w(f, d)
        out["Wu"] = w(f, d)
    elif shape.act == "gelu":
        out["W1"] = w(f, d)
    else:
        raise ValueError(f"unknown activation {shape.act!r}")
    out["Wd"] = w(d, f)
    return out


def make_norm_gains(shape: BlockShape, dtype: str, gen: torch.Generator) -> dict:
    """RMSNorm gains of the pre-norm block variant: g_attn, g_ffn [d_model],
    1 + N(0, 0.25^2) (a trained model's gains sit near 1)."""
    dt = torch_dtype(dtype)
    d = shape.d_model
    return {"g_attn": (1.0 + 0.25 * torch.randn(d, generator=gen)).to(dt),
            "g_ffn": (1.0 + 0.25 * torch.randn(d, generator=gen)).to(dt)}


def make_inputs(wl: Workload, seed: int = 0) -> dict:
    """All tensors of one workload, on the CPU, in the workload's dtype."""
    gen = torch.Generator().manual_seed(seed)
    dt = torch_dtype(wl.dtype)
    out = make_weights(wl.shape, wl.dtype, gen)
    out["X"] = torch.randn(wl.batch, wl.seq, wl.shape.d_model, generator=gen).to(dt)
    if wl.decode:
        sh = (wl.batch, wl.shape.n_heads, wl.cache_len, wl.shape.d_head)
        out["Kcache"] = torch.randn(*sh, generator=gen).to(dt)
        out["Vcache"] = torch.randn(*sh, generator=gen).to(dt)
    return out


def make_matrix(rows: int, cols: int, dtype: str, gen: torch.Generator, std: float = 1.0) -> torch.Tensor:
    """One N(0, std^2) matrix, for the per-call tests."""
    return (torch.randn(rows, cols, generator=gen) * std).to(torch_dtype(dtype))
