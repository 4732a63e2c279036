"""The Python side's argument checks, on the CPU: a tensor reaches the
library only as a raw address, so the binding refuses host tensors and the
runtime refuses tensors of the wrong device, dtype, layout or shape before
any call (the library cannot tell a host address from a device one)."""
import pytest
import torch


@pytest.fixture(scope="module")
def rt():
    import __graft_entry__
    __graft_entry__.build()
    from tensor_transformer_layer_03_b300 import runtime
    return runtime


def test_binding_refuses_host_tensors(rt):
    from tensor_transformer_layer_03_b300 import tp
    assert tp._ptr(None) is None
    with pytest.raises(ValueError, match="CUDA tensor"):
        tp._ptr(torch.zeros(4))


def test_check_tensor(rt):
    cpu = torch.device("cpu")
    x = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    rt.check_tensor(x, "x", torch.bfloat16, cpu, (None, None, 8))
    rt.check_tensor(x, "x", torch.bfloat16, cpu, (2, 3, 8))
    rt.check_tensor(x, "x", torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="dtype"):
        rt.check_tensor(x.float(), "x", torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="contiguous"):
        rt.check_tensor(x.transpose(0, 1), "x", torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="shape"):
        rt.check_tensor(x, "x", torch.bfloat16, cpu, (None, None, 16))
    with pytest.raises(ValueError, match="shape"):
        rt.check_tensor(x, "x", torch.bfloat16, cpu, (None, 8))
    with pytest.raises(ValueError, match="on cpu"):
        rt.check_tensor(x, "x", torch.bfloat16, torch.device("cuda", 0))
    with pytest.raises(TypeError):
        rt.check_tensor([1, 2], "x", torch.bfloat16, cpu)


def test_check_caches(rt):
    cpu = torch.device("cpu")
    k = torch.zeros(3, 4, 10, 16, dtype=torch.bfloat16)
    rt.check_caches(None, None, 2, 4, 16, torch.bfloat16, cpu)
    rt.check_caches(k, k.clone(), 2, 4, 16, torch.bfloat16, cpu)   # more sequences than the call uses
    with pytest.raises(ValueError, match="together"):
        rt.check_caches(k, None, 2, 4, 16, torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="sequences"):
        rt.check_caches(k, k.clone(), 4, 4, 16, torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="shape"):
        rt.check_caches(k, k.clone(), 2, 8, 16, torch.bfloat16, cpu)    # heads
    with pytest.raises(ValueError, match="shape"):
        rt.check_caches(k, k.clone(), 2, 4, 32, torch.bfloat16, cpu)    # head width
    with pytest.raises(ValueError, match="differ"):
        rt.check_caches(k, torch.zeros(3, 4, 12, 16, dtype=torch.bfloat16), 2, 4, 16, torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="dtype"):
        rt.check_caches(k, k.float(), 2, 4, 16, torch.bfloat16, cpu)
