"""GPU parity of split tails: GEMMs whose last, short round of tiles runs as K-range parts
(fp32 partial tiles in the workspace, added in a fixed order by one more launch).

Shapes are picked so that, on a GB300's 152 SMs, the forward down-projection and dX (one
CTA per tile and CTA pairs), dA and dB, and the attention block's QKV, output, dC and dX
GEMMs split; every output is compared with the full fp64 oracle, the launch counter must
show exactly the predicted fixup launches, and results must repeat bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, bf16_chain_tol
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_attn_inputs, make_inputs

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _tile_n(n: int) -> int:
    return 256 if n % 256 == 0 else 128


def _split_rule(TM: int, BN: int, units: int, M: int, N: int, K: int) -> int:
    tiles = -(-M // TM) * -(-N // BN)
    rem = tiles % units
    if rem == 0:
        return 0
    sk = min(units // rem, -(-K // 64) // 16, _lib.mlp_tp_forward_workspace_bytes() // (TM * BN * 4 * rem))
    return 1 if sk >= 2 else 0


def _splits(M: int, N: int, K: int, BN: int, math: bool = False) -> set:
    """The fixup launches (0 or 1) the library's split rule (include/mlp_tp.h, "Split tails")
    can give this GEMM: rounds of `units` tiles, parts of >= 16 k blocks of 64, at most one
    round of parts, within the forward workspace. Two answers where the tile shape depends
    on how many clusters of four CTAs the device can hold."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = BN == 256 and M > 128
    if pairs and N % 512 == 0 and K >= (4096 if math else 2048):  # CTA pairs then take 512-wide
        BN = 512  # tiles (epilogues with math, bias + GELU and GELU', need the longer K)
    TM, units = (256, sms // 2) if pairs else (128, sms)
    out = {_split_rule(TM, BN, units, M, N, K)}
    if BN == 512 and -(-M // 256) % 2 == 0:  # or two pairs per cluster, 512-row tiles
        out.add(_split_rule(512, 512, sms // 4, M, N, K))
    return out


def _sums(*sets) -> set:
    out = {0}
    for s in sets:
        out = {a + b for a in out for b in s}
    return out


def _mlp_fixups(T, h, f, t):
    up = _splits(T, f, h, _tile_n(f // t), math=True)                          # H, G; and dH
    fwd = _sums(up, _splits(T, h, f, _tile_n(h)))                              # Y = G B + b
    bwd = _sums(up, _splits(T, h, f, _tile_n(h)), _splits(h, f, T, _tile_n(f // t)),  # dX, dA
                _splits(f, h, T, _tile_n(h)))                                  # dB
    return fwd, bwd


def _attn_fixups(b, s, h, a):
    T, hd = b * s, a * D
    fwd = _sums(_splits(T, 3 * hd, h, _tile_n(3 * hd)), _splits(T, h, hd, _tile_n(h)))     # QKV, Y
    bwd = _sums(_splits(T, hd, h, _tile_n(hd)), _splits(hd, h, T, _tile_n(h)),             # dC, dWo
                _splits(T, h, 3 * hd, _tile_n(h)), _splits(h, 3 * hd, T, _tile_n(3 * hd)))  # dX, dWqkv
    return fwd, bwd


def _counted(fn):
    n0 = _lib.mlp_tp_launch_count()
    fn()
    return _lib.mlp_tp_launch_count() - n0


# (T, h, f, t): one CTA per tile (T = 128) splitting Y and dX; clusters of two pairs splitting
# Y and dX; CTA pairs splitting dA and dB (K = T); 256-wide pairs splitting the bias + GELU
# (H, G) and GELU' (dH and its column sums for da) GEMMs; clusters of two pairs splitting those
@pytest.mark.parametrize("T,h,f,t", [(128, 1024, 8192, 4), (512, 1024, 4096, 2), (2048, 256, 1024, 2),
                                     (512, 2048, 2048, 2), (512, 4096, 2048, 2)])
def test_mlp_split_tails_match_oracle(T, h, f, t):
    fx_fwd, fx_bwd = _mlp_fixups(T, h, f, t)
    if max(fx_fwd) + max(fx_bwd) == 0:
        pytest.skip("no GEMM of this shape splits on this device's SM count")
    inp = make_inputs(T, h, f, seed=T + h, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    n_fwd = _counted(lambda: block.forward(dev, buf, t))
    n_bwd = _counted(lambda: block.backward(dev, buf, t))
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    assert n_fwd - 2 in fx_fwd and n_bwd - 6 in fx_bwd, (n_fwd, n_bwd, fx_fwd, fx_bwd)
    assert n_fwd + n_bwd > 8  # at least one split tail ran
    ref = oracle.fwd_bwd(inp)
    for k in ("H", "G", "Y", "dX", "dA", "dB", "da", "db"):
        assert_close(k, buf[k], ref[k])
    first = {k: buf[k].clone() for k in ("Y", "dX", "dA", "dB")}
    block.step(dev, buf, t)
    for k, v in first.items():
        assert torch.equal(v, buf[k]), f"{k} differs between two runs"
    # without a forward workspace every tile runs whole: same values up to the sum order
    _lib.mlp_tp_forward(dev["X"], dev["A"], dev["a"], dev["B"], dev["b"], T, h, f, t, buf["H"], buf["G"], buf["Y"],
                        None, 0)
    assert_close("Y (whole tiles)", buf["Y"], ref["Y"])
    rel = float((buf["Y"].double() - first["Y"].double()).norm() / first["Y"].double().norm())
    assert rel < 2e-3, rel


def test_attention_split_tails_match_oracle():
    b, s, h, a, t = 1, 1024, 2048, 16, 2
    fx_fwd, fx_bwd = _attn_fixups(b, s, h, a)
    if max(fx_fwd) + max(fx_bwd) == 0:
        pytest.skip("no GEMM of this shape splits on this device's SM count")
    inp = make_attn_inputs(b, s, h, a, D, seed=11, sw=1.2 / np.sqrt(h), sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_attn_buffers(b, s, h, a, D, t)
    n_fwd = _counted(lambda: block.attn_forward(dev, buf, b, s, a, t, True))
    n_bwd = _counted(lambda: block.attn_backward(dev, buf, b, s, a, t, True))
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    assert n_fwd - 3 in fx_fwd and n_bwd - 7 in fx_bwd, (n_fwd, n_bwd, fx_fwd, fx_bwd)
    assert n_fwd + n_bwd > 10  # at least one split tail ran
    ref = oracle.attn_fwd_bwd({k: v.double().numpy() for k, v in inp.items() if k != "Wqkv"}, b, s, a, True)
    # bf16 roundings on each path, as in the attention parity tests
    for name, n, got, want in (("QKV", 1, buf["QKV"], np.concatenate([ref["Q"], ref["K"], ref["V"]], axis=1)),
                               ("Y", 6, buf["Y"], ref["Y"]), ("dX", 9, buf["dX"], ref["dX"]),
                               ("dWo", 6, buf["dWo"], ref["dWo"])):
        rel, mx = bf16_chain_tol(n)
        assert_close(name, got, want, rel, mx)
    hd = a * D
    dW = buf["dWqkv"].cpu()
    for i, k in enumerate(("dWq", "dWk", "dWv")):
        rel, mx = bf16_chain_tol(9)
        assert_close(k, dW[:, i * hd:(i + 1) * hd], ref[k], rel, mx)
    first = {k: buf[k].clone() for k in ("QKV", "Y", "dX", "dWqkv", "dWo")}
    block.attn_step(dev, buf, b, s, a, t, True)
    for k, v in first.items():
        assert torch.equal(v, buf[k]), f"{k} differs between two runs"


def test_two_pair_clusters_whole_tiles_match_oracle():
    """Several whole 512 x 512 work tiles per cluster of two CTA pairs (B multicast): the
    down-projection and dX are 2 x 36 tiles (two per cluster on a GB300, no split), dA runs on
    CTA pairs; every output against the full oracle, and bit-for-bit repeatable."""
    T, h, f, t = 1024, 18432, 2048, 2
    inp = make_inputs(T, h, f, seed=7, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    block.step(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    ref = oracle.fwd_bwd(inp)
    for k in ("H", "G", "Y", "dX", "dA", "dB", "da", "db"):
        assert_close(k, buf[k], ref[k])
    first = {k: buf[k].clone() for k in ("Y", "dX", "dA", "dB")}
    block.step(dev, buf, t)
    for k, v in first.items():
        assert torch.equal(v, buf[k]), f"{k} differs between two runs"
