"""GPU parity of the backward that recomputes G = GELU(H) instead of keeping the forward's G."""
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


@pytest.mark.parametrize("T,h,f,t", [(128, 64, 256, 2), (300, 200, 800, 2), (512, 512, 2048, 4), (777, 264, 1536, 3),
                                     (2560, 512, 4096, 8)])
def test_backward_with_gelu_recompute(T, h, f, t):
    inp = make_inputs(T, h, f, seed=3, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    block.forward(dev, buf, t)
    block.backward(dev, buf, t)  # the reference: the backward that reads the forward's G
    kept = {k: buf[k].clone() for k in ("dX", "dA", "dB", "da", "db")}
    G_fwd = buf["G"].clone()
    buf["G"].fill_(float("nan"))  # the forward's G was scratch: the recompute must not read it
    ws_bytes = _lib.mlp_tp_recompute_workspace_bytes(T, h, f, t)
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")
    out = {k: torch.full_like(v, float("nan")) for k, v in kept.items()}
    _lib.mlp_tp_backward_recompute(dev["X"], dev["A"], dev["B"], buf["H"], dev["dY"], T, h, f, t, out["dX"],
                                   out["dA"], out["dB"], out["da"], out["db"], ws, ws_bytes)
    assert _lib.mlp_tp_query_device_status() == 0
    for k in ("dX", "dA", "da", "db"):  # these never touch G: bitwise the kept-G backward
        assert torch.equal(out[k], kept[k]), k
    # the forward computes G from the rounded H, as the recompute must: the same G to the bit,
    # hence the same dB
    G_rec = ws[((T * f * 2 + 255) // 256) * 256:][: T * f * 2].view(torch.bfloat16).view(T, f)
    assert torch.equal(G_rec, G_fwd)
    assert torch.equal(out["dB"], kept["dB"])
    ref = oracle.fwd_bwd({k: v.double().numpy() for k, v in inp.items()})
    assert_close("dB", out["dB"], ref["dB"])
    assert_close("G recomputed", G_rec, ref["G"])
    fs = f // t
    for i in range(t):
        assert_close(f"dB shard {i}", out["dB"][i * fs:(i + 1) * fs], ref["dB"][i * fs:(i + 1) * fs])


def test_recompute_rejects_short_workspace():
    T, h, f, t = 64, 64, 128, 1
    inp = make_inputs(T, h, f, seed=1)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    need = _lib.mlp_tp_recompute_workspace_bytes(T, h, f, t)
    assert need > _lib.mlp_tp_workspace_bytes(T, h, f, t)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_backward_recompute(dev["X"], dev["A"], dev["B"], buf["H"], dev["dY"], T, h, f, t, buf["dX"],
                                       buf["dA"], buf["dB"], buf["da"], buf["db"], ws, need - 256)
    assert ei.value.name == "MLP_EWORKSPACE"
