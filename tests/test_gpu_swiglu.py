"""GPU parity of the SwiGLU variant of the block against the fp64 oracle."""
import gc

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, sample_rows_cols
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import WORKLOADS, make_any_inputs, make_swiglu_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _run(inp_cpu, t):
    dev = {k: v.cuda() for k, v in inp_cpu.items()}
    T, h = inp_cpu["X"].shape
    f = inp_cpu["A"].shape[1]
    buf = block.empty_swiglu_buffers(T, h, f, t)
    block.swiglu_step(dev, buf, t)
    st = _lib.mlp_tp_query_device_status()
    assert st == 0, f"device status {st}: {_lib.mlp_tp_last_device_where()}"
    return buf


# single CTAs (128 rows), CTA pairs, ragged T/h/f, several shard counts
@pytest.mark.parametrize("T,h,f,t,sw", [(128, 64, 256, 2, 0.2), (300, 200, 800, 2, 0.1), (512, 512, 2048, 4, 0.05),
                                        (777, 264, 1536, 3, 0.05), (1, 8, 8, 1, 0.2), (2560, 512, 4096, 8, 0.03)])
def test_swiglu_parity_full_oracle(T, h, f, t, sw):
    inp = make_swiglu_inputs(T, h, f, seed=0, sw=sw, sdy=1.0)
    buf = _run(inp, t)
    ref = oracle.swiglu_fwd_bwd(inp)
    for k in ("Ha", "Hg", "U", "Y", "dX", "dA", "dWg", "dB"):
        assert_close(k, buf[k], ref[k])
    fs = f // t
    for i in range(t):
        sl = slice(i * fs, (i + 1) * fs)
        assert_close(f"dA shard {i}", buf["dA"][:, sl], ref["dA"][:, sl])
        assert_close(f"dWg shard {i}", buf["dWg"][:, sl], ref["dWg"][:, sl])
        assert_close(f"dB shard {i}", buf["dB"][sl], ref["dB"][sl])


def test_swiglu_deterministic():
    inp = make_swiglu_inputs(300, 200, 800, seed=4, sw=0.1, sdy=1.0)
    a, b = _run(inp, 2), _run(inp, 2)
    for k in ("Ha", "Hg", "U", "Y", "dX", "dA", "dWg", "dB"):
        assert torch.equal(a[k], b[k]), k


def test_swiglu_full_size_sampled():
    w = WORKLOADS["gpt3-175b-swiglu"]
    inp = make_any_inputs(w)
    buf = _run(inp, w.t)
    rows, cols = sample_rows_cols(w.T, w.f, w.t, n=24)
    rt, ct = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    got = {"Y_rows": buf["Y"][rt], "dX_rows": buf["dX"][rt], "dA_cols": buf["dA"][:, ct],
           "dWg_cols": buf["dWg"][:, ct], "dB_rows": buf["dB"][ct]}
    got = {k: v.cpu() for k, v in got.items()}
    del buf
    gc.collect()
    torch.cuda.empty_cache()
    ref = oracle.swiglu_sampled_bf16(inp, rows, cols)
    for k in got:
        assert_close(f"swiglu {k}", got[k], ref[k])
