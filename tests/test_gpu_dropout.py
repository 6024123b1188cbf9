"""GPU parity of the fused bias + dropout + residual-add output step and its backward.

The keep mask is an integer decision (Philox4x32-10 words against floor(p * 2^24)), taken
the same way on both sides, so the GPU's dropped elements must match the oracle's exactly;
values are compared within the block's tolerance."""
import gc

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, sample_rows_cols
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import WORKLOADS, make_inputs, make_workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _residual(T, h, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn((T, h), generator=g).to(torch.bfloat16)


def _forward_dropout(inp_cpu, R_cpu, t, p, seed, offset):
    dev = {k: v.cuda() for k, v in inp_cpu.items()}
    T, h = inp_cpu["X"].shape
    f = inp_cpu["A"].shape[1]
    buf = block.empty_buffers(T, h, f, t)
    R = R_cpu.cuda()
    Z = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    _lib.mlp_tp_forward_residual_dropout(dev["X"], dev["A"], dev["a"], dev["B"], dev["b"], R, T, h, f, t, p, seed,
                                         offset, buf["H"], buf["G"], Z)
    return dev, buf, Z


@pytest.mark.parametrize("T,h,f,t,p", [(128, 64, 256, 2, 0.1), (300, 200, 800, 2, 0.5), (512, 512, 2048, 4, 0.1),
                                       (777, 264, 1536, 3, 0.0), (64, 8, 8, 1, 0.9)])
def test_forward_backward_with_dropout_matches_oracle(T, h, f, t, p):
    seed, offset = 1234 + T, 7
    inp = make_inputs(T, h, f, seed=1, sdy=1.0)
    R = _residual(T, h, seed=5)
    dev, buf, Z = _forward_dropout(inp, R, t, p, seed, offset)
    dZ = inp["dY"].cuda()  # the upstream gradient of Z
    dY = torch.empty_like(dZ)
    _lib.mlp_tp_dropout_backward(dZ, T, h, p, seed, offset, dY)
    dev["dY"] = dY
    block.backward(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0
    ref = oracle.fwd_bwd_residual_dropout(inp, R, inp["dY"], p, seed, offset)
    keep = ref["keep"].astype(bool)
    # dropped elements: dY is exactly zero there, and only there (dZ has no zeros)
    got_zero = (dY.cpu() == 0).numpy()
    np.testing.assert_array_equal(got_zero, ~keep)
    for k, g in (("Z", Z), ("H", buf["H"]), ("G", buf["G"]), ("dY", dY), ("dX", buf["dX"]), ("dA", buf["dA"]),
                 ("da", buf["da"]), ("dB", buf["dB"]), ("db", buf["db"])):
        assert_close(k, g, ref[k])


def test_dropped_outputs_equal_the_residual_exactly():
    """With R = 0 a dropped element of Z is exactly 0; kept ones are (almost surely) not."""
    T, h, f, t, p, seed = 256, 512, 1024, 2, 0.3, 99
    inp = make_inputs(T, h, f, seed=2, sdy=1.0)
    R = torch.zeros((T, h), dtype=torch.bfloat16)
    _, _, Z = _forward_dropout(inp, R, t, p, seed, 0)
    keep = oracle.dropout_keep(T, h, p, seed, 0).astype(bool)
    z = Z.cpu().float().numpy()
    assert np.all(z[~keep] == 0.0)
    assert np.mean(z[keep] != 0.0) > 0.999


def test_seed_and_offset_change_the_mask():
    T, h = 64, 256
    dZ = torch.ones((T, h), dtype=torch.bfloat16, device="cuda")
    outs = []
    for seed, offset in ((1, 0), (1, 1), (2, 0), (1, 0)):
        dY = torch.empty_like(dZ)
        _lib.mlp_tp_dropout_backward(dZ, T, h, 0.5, seed, offset, dY)
        outs.append(dY.cpu())
    assert torch.equal(outs[0], outs[3])
    assert not torch.equal(outs[0], outs[1]) and not torch.equal(outs[0], outs[2])
    for o, (seed, offset) in zip(outs, ((1, 0), (1, 1), (2, 0), (1, 0))):
        np.testing.assert_array_equal((o != 0).numpy(), oracle.dropout_keep(T, h, 0.5, seed, offset).astype(bool))


def test_rejects_bad_probability():
    T, h = 8, 16
    buf = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    for p in (-0.1, 1.0, float("nan")):
        with pytest.raises(_lib.MlpError) as ei:
            _lib.mlp_tp_dropout_backward(buf, T, h, p, 0, 0, buf)
        assert ei.value.name == "MLP_EINVAL"


def test_full_size_gpt3_175b_sampled_rows():
    w = WORKLOADS["gpt3-175b"]
    p, seed, offset = 0.1, 2024, 3
    inp = make_workload_inputs(w)
    R = _residual(w.T, w.h, seed=11)
    dev, buf, Z = _forward_dropout(inp, R, w.t, p, seed, offset)
    assert _lib.mlp_tp_query_device_status() == 0
    rows, cols = sample_rows_cols(w.T, w.f, w.t)
    Zr = Z[torch.from_numpy(rows).cuda()].cpu()
    del dev, buf, Z
    gc.collect()
    torch.cuda.empty_cache()
    ref = oracle.sampled_bf16(inp, rows, cols[:2])
    keep = oracle.dropout_keep(w.T, w.h, p, seed, offset)[rows]
    Zref = oracle.residual_dropout(ref["Y_rows"], R[torch.from_numpy(rows)], keep, p)
    assert_close("Z rows", Zr, Zref)
    Rr = R[torch.from_numpy(rows)].float().numpy()
    np.testing.assert_array_equal(Zr.float().numpy()[~keep.astype(bool)], Rr[~keep.astype(bool)])
