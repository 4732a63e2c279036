"""The seeded input recipe that both the oracle and the library consume:
one CPU generator seeded per workload, fp32 randn drawn in the order Wq, Wk,
Wv, Wo, (Wg, Wu | W1), Wd, X, [Kcache, Vcache], weights scaled by 0.02, then
a cast to the workload dtype; the same seed gives the same tensors."""
import torch

from tensor_transformer_layer_03_b300 import inputs as I


def _recipe(wl, seed):
    g = torch.Generator().manual_seed(seed)
    dt = I.torch_dtype(wl.dtype)
    d, f = wl.shape.d_model, wl.shape.d_ffn
    names = ["Wq", "Wk", "Wv", "Wo"] + (["Wg", "Wu"] if wl.shape.act == "swiglu" else ["W1"]) + ["Wd"]
    shapes = {"Wq": (d, d), "Wk": (d, d), "Wv": (d, d), "Wo": (d, d), "Wg": (f, d), "Wu": (f, d), "W1": (f, d),
              "Wd": (d, f)}
    out = {n: (torch.randn(*shapes[n], generator=g) * 0.02).to(dt) for n in names}
    out["X"] = torch.randn(wl.batch, wl.seq, d, generator=g).to(dt)
    if wl.decode:
        sh = (wl.batch, wl.shape.n_heads, wl.cache_len, wl.shape.d_head)
        out["Kcache"] = torch.randn(*sh, generator=g).to(dt)
        out["Vcache"] = torch.randn(*sh, generator=g).to(dt)
    return out


def test_recipe_matches_the_stated_order():
    for wl in (I.WORKLOADS["tiny_fp32"],
               I.Workload("small_decode", I.BlockShape(256, 4, 512, "swiglu"), tp=2, batch=2, seq=1, causal=True,
                          dtype="bf16", decode=True, cache_len=9)):
        got = I.make_inputs(wl, seed=3)
        ref = _recipe(wl, 3)
        assert sorted(got) == sorted(ref)
        for k in ref:
            assert got[k].dtype == ref[k].dtype and torch.equal(got[k], ref[k]), k


def test_same_seed_same_tensors_other_seed_differs():
    wl = I.WORKLOADS["tiny_fp32"]
    a, b, c = I.make_inputs(wl, 0), I.make_inputs(wl, 0), I.make_inputs(wl, 1)
    assert all(torch.equal(a[k], b[k]) for k in a)
    assert not torch.equal(a["X"], c["X"])


def test_norm_gains_near_one():
    g = torch.Generator().manual_seed(0)
    gains = I.make_norm_gains(I.LLAMA7B, "bf16", g)
    for v in gains.values():
        v = v.float()
        assert v.shape == (4096,) and abs(v.mean().item() - 1.0) < 0.02 and 0.2 < v.std().item() < 0.3
