"""GPU parity of the GELU recompute, in which G = GELU(H) is never stored: the forward keeps H
alone and its down-projection reads H, turning each A tile into G in shared memory; the
backward's dB GEMM does the same. G there is the forward epilogue's G bit for bit, so the
forward's Y and every gradient must equal those of the path that keeps G, bit for bit, and
match the fp64 oracle."""
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


# one CTA per tile; ragged pairs; 256-wide pairs; odd shard counts; 512-wide tiles on clusters of
# two CTA pairs for the down-projection (N = h, K = f) and dB (N = h, K = T); split tails
SHAPES = [(128, 64, 256, 2), (300, 200, 800, 2), (512, 512, 2048, 4), (777, 264, 1536, 3), (2560, 512, 4096, 8),
          (2048, 1024, 4096, 2), (512, 1024, 4096, 2), (2048, 256, 1024, 2)]


@pytest.mark.parametrize("T,h,f,t", SHAPES, ids=[f"T{T}-h{h}-f{f}-t{t}" for T, h, f, t in SHAPES])
def test_recompute_forward_and_backward(T, h, f, t):
    inp = make_inputs(T, h, f, seed=3, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    block.step(dev, buf, t)  # the reference: the path that keeps G
    kept = {k: buf[k].clone() for k in ("H", "Y", "dX", "dA", "dB", "da", "db")}
    fws = torch.empty((_lib.mlp_tp_forward_workspace_bytes(),), dtype=torch.uint8, device="cuda")

    H = torch.full((T, f), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((T, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    _lib.mlp_tp_forward_recompute(dev["X"], dev["A"], dev["a"], dev["B"], dev["b"], T, h, f, t, H, Y, fws,
                                  fws.numel())
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    assert torch.equal(H, kept["H"]), "H differs from the forward that keeps G"
    assert torch.equal(Y, kept["Y"]), "Y differs from the forward that keeps G"

    ws_bytes = _lib.mlp_tp_recompute_workspace_bytes(T, h, f, t)
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")
    out = {k: torch.full_like(kept[k], float("nan")) for k in ("dX", "dA", "dB", "da", "db")}
    _lib.mlp_tp_backward_recompute(dev["X"], dev["A"], dev["B"], H, dev["dY"], T, h, f, t, out["dX"], out["dA"],
                                   out["dB"], out["da"], out["db"], ws, ws_bytes)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    for k in ("dX", "dA", "dB", "da", "db"):
        assert torch.equal(out[k], kept[k]), f"{k} differs from the backward that keeps G"

    ref = oracle.fwd_bwd(inp)
    for k, v in (("H", H), ("Y", Y), ("dB", out["dB"]), ("dX", out["dX"]), ("da", out["da"])):
        assert_close(k, v, ref[k])
    fs = f // t
    for i in range(t):
        assert_close(f"dB shard {i}", out["dB"][i * fs:(i + 1) * fs], ref["dB"][i * fs:(i + 1) * fs])


def test_recompute_is_deterministic():
    T, h, f, t = 2048, 1024, 4096, 2
    inp = make_inputs(T, h, f, seed=9, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    ws_bytes = _lib.mlp_tp_recompute_workspace_bytes(T, h, f, t)
    runs = []
    for _ in range(2):
        H = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
        Y = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")
        g = {"dX": torch.empty((T, h), dtype=torch.bfloat16, device="cuda"),
             "dA": torch.empty((h, f), dtype=torch.bfloat16, device="cuda"),
             "dB": torch.empty((f, h), dtype=torch.bfloat16, device="cuda"),
             "da": torch.empty((f,), device="cuda"), "db": torch.empty((h,), device="cuda")}
        _lib.mlp_tp_forward_recompute(dev["X"], dev["A"], dev["a"], dev["B"], dev["b"], T, h, f, t, H, Y, ws,
                                      ws_bytes)
        _lib.mlp_tp_backward_recompute(dev["X"], dev["A"], dev["B"], H, dev["dY"], T, h, f, t, g["dX"], g["dA"],
                                       g["dB"], g["da"], g["db"], ws, ws_bytes)
        assert _lib.mlp_tp_query_device_status() == 0
        runs.append(dict(g, Y=Y))
    for k in runs[0]:
        assert torch.equal(runs[0][k], runs[1][k]), k


def test_recompute_rejects_short_workspace():
    T, h, f, t = 64, 64, 128, 1
    inp = make_inputs(T, h, f, seed=1)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    need = _lib.mlp_tp_recompute_workspace_bytes(T, h, f, t)
    assert need == _lib.mlp_tp_workspace_bytes(T, h, f, t)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_backward_recompute(dev["X"], dev["A"], dev["B"], buf["H"], dev["dY"], T, h, f, t, buf["dX"],
                                       buf["dA"], buf["dB"], buf["da"], buf["db"], ws, need - 256)
    assert ei.value.name == "MLP_EWORKSPACE"
