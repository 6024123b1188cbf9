"""The allocation-free bias-gradient entry point, for callers that cannot allocate device
memory when they need da and db (code inside another runtime that owns all device memory,
or latency-bound loops where cudaMalloc would synchronise the device). It must give the
same sums as mlp_tp_backward, call after call, while its partial sums live in the
library's fixed device array instead of a workspace.

This file is collected last on purpose, so a run that stops at the first failure has
already run every other test."""
import pytest
import torch

from parity import assert_close
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _backward_reference(T, h, f, t, seed):
    inp = {k: v.cuda() for k, v in make_inputs(T, h, f, seed=seed, sdy=1.0).items()}
    buf = block.empty_buffers(T, h, f, t)
    block.step(inp, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0
    # mlp_tp_backward leaves dH in the first T*f*2 bytes of its workspace
    dH = buf["ws"][: T * f * 2].view(torch.bfloat16).view(T, f)
    return inp, buf, dH


@pytest.mark.parametrize("T,h,f,t", [(128, 64, 256, 2), (1000, 200, 800, 2), (4096, 512, 2048, 4)])
def test_noalloc_matches_backward_on_two_calls_in_a_row(T, h, f, t):
    inp, buf, dH = _backward_reference(T, h, f, t, seed=T)
    for call in range(2):
        da = torch.full((f,), float("nan"), device="cuda")
        db = torch.full((h,), float("nan"), device="cuda")
        _lib.mlp_tp_bias_grads_noalloc(dH, inp["dY"], T, h, f, da, db)
        assert _lib.mlp_tp_query_device_status() == 0
        assert_close(f"da call {call}", da, buf["da"].double().cpu().numpy())
        assert_close(f"db call {call}", db, buf["db"].double().cpu().numpy())


def test_noalloc_consecutive_sizes_do_not_leak_state():
    """A large call, then a small one: the small one must not read the large one's partials."""
    big = _backward_reference(4096, 512, 2048, 4, seed=1)
    small = _backward_reference(600, 64, 128, 1, seed=2)
    for inp, buf, dH in (big, small):
        T, h = inp["dY"].shape
        f = dH.shape[1]
        da = torch.empty(f, device="cuda")
        db = torch.empty(h, device="cuda")
        _lib.mlp_tp_bias_grads_noalloc(dH, inp["dY"], T, h, f, da, db)
        assert_close("da", da, buf["da"].double().cpu().numpy())
        assert_close("db", db, buf["db"].double().cpu().numpy())


def test_noalloc_rejects_sizes_beyond_its_array():
    # 16 row slices x (f + h) columns must fit in 2^20 floats
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_bias_grads_noalloc(0x10000, 0x10000, 16384, 8192, 65536, 0x10000, 0x10000)
    assert ei.value.name == "MLP_EWORKSPACE"
