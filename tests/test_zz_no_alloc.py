"""The allocation-free bias-gradient entry point, for callers that cannot allocate device
memory when they need da and db: code inside another runtime that owns all device memory
(a framework's caching allocator, or a fixed arena with nothing left to lend), and
latency-bound loops where a cudaMalloc would synchronise the device. Its partial sums live
in the library's fixed device array instead of a workspace.

Checked on two calls in a row: da and db against the fp64 oracle's, db bit for bit
against mlp_tp_backward's (the same reduction over dY in the same order), and da against
mlp_tp_backward's within the tolerance (this entry point sums the bf16 dH it is given; the
backward sums the dH GEMM's fp32 values before they are rounded).

This file is collected last on purpose, so a run that stops at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import oracle
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
    cpu = make_inputs(T, h, f, seed=seed, sdy=1.0)
    inp = {k: v.cuda() for k, v in cpu.items()}
    buf = block.empty_buffers(T, h, f, t)
    block.step(inp, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0
    # mlp_tp_backward leaves dH in the first T*f*2 bytes of its workspace
    dH = buf["ws"][: T * f * 2].view(torch.bfloat16).view(T, f)
    ref = oracle.fwd_bwd(cpu)
    return inp, buf, dH, ref


def _check(inp, buf, dH, ref, T, h, f, what):
    da = torch.full((f,), float("nan"), device="cuda")
    db = torch.full((h,), float("nan"), device="cuda")
    _lib.mlp_tp_bias_grads_noalloc(dH, inp["dY"], T, h, f, da, db)
    assert _lib.mlp_tp_query_device_status() == 0
    assert_close(f"da {what} vs oracle", da, ref["da"])
    assert_close(f"db {what} vs oracle", db, ref["db"])
    assert torch.equal(db, buf["db"]), f"db {what}: not bitwise mlp_tp_backward's"
    assert_close(f"da {what} vs mlp_tp_backward", da, buf["da"].double().cpu().numpy())
    assert np.isfinite(da.cpu().numpy()).all()


@pytest.mark.parametrize("T,h,f,t", [(128, 64, 256, 2), (1000, 200, 800, 2), (4096, 512, 2048, 4)])
def test_noalloc_matches_oracle_and_backward_on_two_calls_in_a_row(T, h, f, t):
    inp, buf, dH, ref = _backward_reference(T, h, f, t, seed=T)
    for call in range(2):
        _check(inp, buf, dH, ref, T, h, f, f"call {call}")


def test_noalloc_consecutive_sizes_do_not_leak_state():
    """A large call, then a small one: the small one must not read the large one's partials."""
    for (T, h, f, t, seed) in ((4096, 512, 2048, 4, 1), (600, 64, 128, 1, 2)):
        inp, buf, dH, ref = _backward_reference(T, h, f, t, seed=seed)
        _check(inp, buf, dH, ref, T, h, f, f"T={T}")


def test_noalloc_rejects_sizes_beyond_its_array():
    # 16 row slices x (f + h) columns must fit in 2^20 floats
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_bias_grads_noalloc(0x10000, 0x10000, 16384, 8192, 65536, 0x10000, 0x10000)
    assert ei.value.name == "MLP_EWORKSPACE"
