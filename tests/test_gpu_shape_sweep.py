"""GPU parity over a seeded sweep of MLP block shapes, against the full fp64 oracle.

The shapes are drawn to reach every branch of the GEMM launch planner on a GB300 (152 SMs):
128-, 256- and 512-wide tiles; one CTA per tile, CTA pairs and clusters of two pairs; whole
rounds and split tails; and ragged edges in every GEMM dimension, for each epilogue (bias +
GELU, GELU' with its column sums, bias, plain). Three families:
  ragged  T, h and f/t any multiples of 8 (T any), t from 1 to 8;
  wide    h or f a multiple of 512 with K long enough for 512-wide tiles (K = T for dA and
          dB), an odd or even number of 256-row blocks (pairs or clusters), the last one
          partly filled;
  short   at most 256 tokens against long K, so most tiles run as split parts, and at most
          128 tokens with K too short to split.
Every output (H, G, Y, dX, dA, dB, da, db) is compared element by element. A second sweep does
the same for the attention block: sequence lengths off the 128-query and 64-key blocks, several
sequences and heads per shard, causal and unmasked."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, bf16_chain_tol
from sweep_shapes import attn_sweep_shapes, mlp_sweep_shapes
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_attn_inputs, make_inputs

pytestmark = pytest.mark.gpu


SHAPES = mlp_sweep_shapes()


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


@pytest.mark.parametrize("T,h,f,t", SHAPES, ids=[f"T{T}-h{h}-f{f}-t{t}" for T, h, f, t in SHAPES])
def test_shape_sweep_matches_oracle(T, h, f, t):
    inp = make_inputs(T, h, f, seed=T + h + f + t, sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_buffers(T, h, f, t)
    block.step(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    ref = oracle.fwd_bwd(inp)
    for k in ("H", "G", "Y", "dX", "dA", "dB", "da", "db"):
        assert_close(k, buf[k], ref[k])


D = 128
# bf16 roundings on each attention output's path (as in the attention parity tests)
ATTN_ROUNDINGS = {"QKV": 1, "C": 4, "L": 2, "Y": 6, "dX": 9, "dWq": 9, "dWk": 9, "dWv": 7, "dWo": 6}


ATTN_SHAPES = attn_sweep_shapes()


@pytest.mark.parametrize("b,s,h,a,t,causal", ATTN_SHAPES,
                         ids=[f"b{b}-s{s}-h{h}-a{a}-t{t}-{'causal' if c else 'full'}" for b, s, h, a, t, c in ATTN_SHAPES])
def test_attention_shape_sweep_matches_oracle(b, s, h, a, t, causal):
    inp = make_attn_inputs(b, s, h, a, D, seed=b + s + h + a, sw=1.2 / np.sqrt(h), sdy=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_attn_buffers(b, s, h, a, D, t)
    block.attn_step(dev, buf, b, s, a, t, causal)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    ref = oracle.attn_fwd_bwd({k: v.double().numpy() for k, v in inp.items() if k != "Wqkv"}, b, s, a, causal)

    def close(name, gpu, want):
        rel, mx = bf16_chain_tol(ATTN_ROUNDINGS[name])
        assert_close(name, gpu, want, rel, mx)

    close("QKV", buf["QKV"], np.concatenate([ref["Q"], ref["K"], ref["V"]], axis=1))
    for k in ("C", "L", "Y", "dX", "dWo"):
        close(k, buf[k], ref[k])
    hd = a * D
    dW = buf["dWqkv"].cpu()
    for i, k in enumerate(("dWq", "dWk", "dWv")):
        close(k, dW[:, i * hd:(i + 1) * hd], ref[k])
