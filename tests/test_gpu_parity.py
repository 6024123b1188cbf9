"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small and ragged shapes are checked element by element against the full oracle; the
full-size GPT layer workloads are checked on sampled entries that the oracle computes
exactly (rows of Y and dX; columns of dA, rows of dB and entries of da, including the
first and last column of every shard; all of db)."""
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


def _run(inp_cpu: dict, t: int):
    dev = {k: v.cuda() for k, v in inp_cpu.items()}
    T, h = inp_cpu["X"].shape
    f = inp_cpu["A"].shape[1]
    buf = block.empty_buffers(T, h, f, t)
    block.step(dev, buf, t)
    st = _lib.mlp_tp_query_device_status()
    assert st == 0, f"device status {st}: {_lib.mlp_tp_last_device_where()}"
    return dev, buf


def _check_full(inp_cpu: dict, buf: dict, t: int, ref: dict) -> None:
    f = inp_cpu["A"].shape[1]
    fs = f // t
    for k in ("H", "G", "Y", "dX", "dA", "dB", "da", "db"):
        assert_close(k, buf[k], ref[k])
    for i in range(t):  # per shard slice, so one bad shard cannot hide in the whole
        sl = slice(i * fs, (i + 1) * fs)
        assert_close(f"dA shard {i}", buf["dA"][:, sl], ref["dA"][:, sl])
        assert_close(f"dB shard {i}", buf["dB"][sl], ref["dB"][sl])
        assert_close(f"da shard {i}", buf["da"][sl], ref["da"][sl])
        assert_close(f"G shard {i}", buf["G"][:, sl], ref["G"][:, sl])


# (T, h, f, t, sdy): several tiles, ragged tails in every GEMM dimension, both tile widths
SMALL = [
    (128, 64, 256, 2, 1.0),     # the tiny workload's shape
    (128, 64, 256, 1, 1.0),
    (128, 64, 256, 8, 1.0),
    (300, 200, 800, 2, 1.0),    # T, h, f/t not multiples of the tile sizes
    (1, 8, 8, 1, 1.0),          # one token, smallest legal widths
    (130, 136, 520, 5, 1.0),    # f/t = 104: shard edges inside tiles
    (512, 512, 2048, 4, 0.01),  # f/t = 512: 256-wide tiles, several K blocks
    (777, 264, 1536, 3, 0.01),
]


@pytest.mark.parametrize("T,h,f,t,sdy", SMALL)
def test_parity_full_oracle(T, h, f, t, sdy):
    inp = make_inputs(T, h, f, seed=0, sdy=sdy)
    _, buf = _run(inp, t)
    ref = oracle.fwd_bwd(inp)
    _check_full(inp, buf, t, ref)


def test_tiny_workload_every_shard_count():
    w = WORKLOADS["tiny"]
    inp = make_workload_inputs(w)
    ref = oracle.fwd_bwd(inp)
    for t in (1, 2, 4, 8, 16, 32):
        _, buf = _run(inp, t)
        _check_full(inp, buf, t, ref)


def test_deterministic_bitwise():
    inp = make_inputs(300, 200, 800, seed=5, sdy=1.0)
    _, b1 = _run(inp, 2)
    _, b2 = _run(inp, 2)
    for k in ("H", "G", "Y", "dX", "dA", "dB", "da", "db"):
        assert torch.equal(b1[k], b2[k]), k


def test_no_tokens():
    h, f, t = 64, 256, 2
    inp = make_inputs(0, h, f, seed=0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(0, h, f, t)
    for k in ("dA", "dB", "da", "db"):
        buf[k].fill_(7)
    block.step(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0
    for k in ("dA", "dB", "da", "db"):
        assert torch.count_nonzero(buf[k]) == 0, k


def test_bounded_wait_reports_timeout_and_context_survives():
    _lib.mlp_tp_selftest_wait_timeout(2_000_000)  # 2 ms; nothing ever completes the barrier
    assert _lib.mlp_tp_query_device_status() == _lib.STATUS_CODES["MLP_ETIMEOUT"]
    assert _lib.mlp_tp_last_device_code() == 6
    assert _lib.mlp_tp_query_device_status() == 0  # cleared by the query
    inp = make_inputs(128, 64, 256, seed=0, sdy=1.0)  # the context still computes
    _, buf = _run(inp, 2)
    assert_close("Y", buf["Y"], oracle.fwd_bwd(inp)["Y"])


def test_gpu_rejects_bad_arguments():
    inp = {k: v.cuda() for k, v in make_inputs(128, 64, 256, seed=0).items()}
    buf = block.empty_buffers(128, 64, 256, 2)
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], 128, 64, 256, 3,
                            buf["H"], buf["G"], buf["Y"], None, 0)
    assert ei.value.name == "MLP_ESHAPE"
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_forward(inp["X"].data_ptr() + 2, inp["A"], inp["a"], inp["B"], inp["b"], 128, 64,
                            256, 2, buf["H"], buf["G"], buf["Y"], None, 0)
    assert ei.value.name == "MLP_EALIGN"
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_backward(inp["X"], inp["A"], inp["B"], buf["H"], buf["G"], inp["dY"], 128, 64, 256, 2,
                             buf["dX"], buf["dA"], buf["dB"], buf["da"], buf["db"], buf["ws"], 64)
    assert ei.value.name == "MLP_EWORKSPACE"


# ---- full-size GPT layer workloads, sampled entries --------------------------------------

BIG = ["gpt-1.7b-t1", "gpt-1.7b-t2", "gpt-18b", "gpt3-175b", "gpt-1t"]


@pytest.mark.parametrize("name", BIG)
def test_parity_full_size_sampled(name):
    w = WORKLOADS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 2 * (4 * w.h * w.f + 6 * w.T * w.f + 6 * w.T * w.h)
    if need > 0.9 * free:
        pytest.skip(f"needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    inp = make_workload_inputs(w)
    dev, buf = _run(inp, w.t)
    rows, cols = sample_rows_cols(w.T, w.f, w.t)
    rows_t, cols_t = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    got = {"Y_rows": buf["Y"][rows_t], "dX_rows": buf["dX"][rows_t], "dA_cols": buf["dA"][:, cols_t],
           "dB_rows": buf["dB"][cols_t], "da": buf["da"][cols_t], "db": buf["db"]}
    got = {k: v.cpu() for k, v in got.items()}
    del dev, buf
    gc.collect()
    torch.cuda.empty_cache()
    ref = oracle.sampled_bf16(inp, rows, cols)
    for k in got:
        assert_close(f"{name} {k}", got[k], ref[k])
    fs = w.f // w.t
    for i in range(w.t):  # shard edges and the sampled columns inside each shard
        m = (cols >= i * fs) & (cols < (i + 1) * fs)
        assert m.sum() >= 2
        assert_close(f"{name} dA shard {i}", got["dA_cols"][:, m], ref["dA_cols"][:, m])
        assert_close(f"{name} dB shard {i}", got["dB_rows"][m], ref["dB_rows"][m])
