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
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_attn_inputs, make_inputs

pytestmark = pytest.mark.gpu


def _sweep_shapes():
    rng = np.random.default_rng(20240611)
    out = []
    while len(out) < 8:  # ragged: small enough that the oracle takes well under a second
        t = int(rng.integers(1, 9))
        T = int(rng.integers(1, 1200))
        h = 8 * int(rng.integers(1, 200))
        f = t * 8 * int(rng.integers(1, 120))
        if T * h * f <= 3e8:
            out.append((T, h, f, t))

    def ragged_rows(blocks):  # blocks 256-row blocks, the last one partly filled
        return 256 * blocks - 8 * int(rng.integers(1, 32))

    for blocks in (2, 3, 4):  # wide down-projection and dX: N = h, K = f >= 2048; clusters or pairs
        t = int(rng.choice([1, 2, 4]))
        out.append((ragged_rows(blocks), 512 * int(rng.integers(1, 3)), 512 * int(rng.integers(4, 7)), t))
    # 39 whole 512-wide tiles on 76 CTA pairs: more than half a round, so no split
    out.append((ragged_rows(3), 512 * 13, 2048, 2))
    for blocks in (3, 4):  # wide up-projection and dH: N = f, K = h >= 4096
        t = int(rng.choice([1, 2]))
        out.append((ragged_rows(blocks), 4096 + 8 * int(rng.integers(0, 64)), 512 * int(rng.integers(1, 3)), t))
    # wide dA and dB (K = T >= 2048): h of two 256-row blocks (clusters) and of three (pairs)
    out.append((2048 + 8 * int(rng.integers(1, 32)), 512, 1024, 2))
    out.append((2048 + 8 * int(rng.integers(1, 32)), 768, 1536, 3))
    for _ in range(2):  # short: few tokens, long K
        t = int(rng.choice([2, 4]))
        T = int(rng.integers(1, 257))
        h = 1024 * int(rng.integers(1, 3))
        f = 2048 * int(rng.integers(2, 4))
        out.append((T, h, f, t))
    # at most 128 tokens, 256-wide tiles, K too short to split
    out.append((int(rng.integers(1, 129)), 256, 512, 2))
    return out


SHAPES = _sweep_shapes()


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


def _attn_shapes():
    """(b, s, h, a, t, causal): any sequence length (ragged query and key blocks, shorter than
    a block), one to three sequences, one to three heads per shard, either mask."""
    rng = np.random.default_rng(20240612)
    out = []
    for i in range(6):
        t = int(rng.integers(1, 4))
        a = t * int(rng.integers(1, 4))
        out.append((int(rng.integers(1, 4)), int(rng.integers(1, 1600)), 8 * int(rng.integers(16, 80)), a, t,
                    bool(i % 3 != 2)))
    return out


ATTN_SHAPES = _attn_shapes()


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
