"""GPU parity of the head-parallel attention block (QKV projection, fused causal attention
core, output projection with the on-chip head-shard sum, and the backward) against the
fp64 oracle."""
import gc

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, bf16_chain_tol
from megatron_tensor_transformer_tcgen05_gb300 import block, _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import ATTN_WORKLOADS, make_attn_inputs, make_attn_workload_inputs

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _run(inp_cpu, b, s, a, t, causal):
    dev = {k: v.cuda() for k, v in inp_cpu.items()}
    h = inp_cpu["X"].shape[1]
    buf = block.empty_attn_buffers(b, s, h, a, D, t)
    block.attn_step(dev, buf, b, s, a, t, causal)
    st = _lib.mlp_tp_query_device_status()
    assert st == 0, f"device status {st}: {_lib.mlp_tp_last_device_where()}"
    return buf


# bf16 roundings on each output's path (the inputs are exact bf16 values):
#   QKV: its own store. C: Q and K (through the scores), V, P (the MMA operand), C.
#   L: Q and K. Y: C's four, C as stored, Y. dX, dWq, dWk: Q, K, V, P, C, dC, dS, dQ/dK, the
#   output. dWv: as those without dS and with P^T in its place. dWo: C's four, C, dWo.
ROUNDINGS = {"QKV": 1, "C": 4, "L": 2, "Y": 6, "dX": 9, "dWq": 9, "dWk": 9, "dWv": 7, "dWo": 6}


def _close(name, gpu, ref):
    rel, mx = bf16_chain_tol(ROUNDINGS[name.split()[0]])
    assert_close(name, gpu, ref, rel, mx)


def _oracle(inp_cpu, b, s, a, causal):
    return oracle.attn_fwd_bwd({k: v.double().numpy() for k, v in inp_cpu.items() if k != "Wqkv"}, b, s, a, causal)


# one block; ragged s; unmasked; s shorter than a block; one token; several shards and
# blocks; more heads than shards
@pytest.mark.parametrize("b,s,h,a,t,causal", [(1, 128, 128, 1, 1, True), (2, 200, 256, 2, 2, True),
                                              (1, 384, 256, 2, 1, False), (2, 64, 128, 1, 1, True),
                                              (1, 1, 128, 1, 1, True), (3, 257, 384, 3, 3, True),
                                              (1, 1024, 512, 4, 2, True), (2, 300, 256, 2, 1, False)])
def test_attention_parity_full_oracle(b, s, h, a, t, causal):
    inp = make_attn_inputs(b, s, h, a, D, seed=s + h, sw=1.2 / np.sqrt(h), sdy=1.0)
    buf = _run(inp, b, s, a, t, causal)
    ref = _oracle(inp, b, s, a, causal)
    _close("QKV", buf["QKV"], np.concatenate([ref["Q"], ref["K"], ref["V"]], axis=1))
    _close("C", buf["C"], ref["C"])
    _close("L", buf["L"], ref["L"])
    _close("Y", buf["Y"], ref["Y"])
    _close("dX", buf["dX"], ref["dX"])
    dW = buf["dWqkv"].cpu()
    hd = a * D
    for i, k in enumerate(("dWq", "dWk", "dWv")):
        _close(k, dW[:, i * hd:(i + 1) * hd], ref[k])
    _close("dWo", buf["dWo"], ref["dWo"])


def test_attention_is_deterministic_and_shard_count_free():
    b, s, h, a = 2, 320, 512, 4
    inp = make_attn_inputs(b, s, h, a, D, seed=5, sw=1.2 / np.sqrt(h), sdy=1.0)
    outs = [_run(inp, b, s, a, t, True) for t in (1, 2, 4, 1)]
    for k in ("Y", "C", "L", "dX", "dWqkv", "dWo"):
        assert torch.equal(outs[0][k], outs[3][k]), k  # bitwise, run to run
        for o in outs[1:3]:
            assert torch.equal(outs[0][k], o[k]), k  # one accumulator whatever the shard count


def test_no_tokens_zeroes_weight_gradients():
    h, a = 256, 2
    inp = make_attn_inputs(1, 8, h, a, D, seed=1)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_attn_buffers(0, 8, h, a, D, 1)
    buf["dWqkv"].fill_(1.0)
    buf["dWo"].fill_(1.0)
    _lib.mlp_tp_attn_forward(None, dev["Wqkv"], dev["Wo"], 0, 8, h, a, D, 1, True, None, None, None, None, None, 0)
    _lib.mlp_tp_attn_backward(None, dev["Wqkv"], dev["Wo"], None, None, None, None, 0, 8, h, a, D, 1, True, None,
                              buf["dWqkv"], buf["dWo"], buf["ws"], buf["ws"].numel())
    assert not buf["dWqkv"].any() and not buf["dWo"].any()


def test_rejects_bad_arguments():
    b, s, h, a = 1, 64, 256, 2
    inp = make_attn_inputs(b, s, h, a, D, seed=1)
    dev = {k: v.cuda() for k, v in inp.items()}
    buf = block.empty_attn_buffers(b, s, h, a, D, 1)

    def fwd(**kw):
        args = dict(b=b, s=s, h=h, a=a, d=D, t=1, X=dev["X"], QKV=buf["QKV"])
        args.update(kw)
        _lib.mlp_tp_attn_forward(args["X"], dev["Wqkv"], dev["Wo"], args["b"], args["s"], args["h"], args["a"],
                                 args["d"], args["t"], True, args["QKV"], buf["C"], buf["L"], buf["Y"], None, 0)

    for kw, name in ((dict(d=64), "MLP_ESHAPE"), (dict(t=3), "MLP_ESHAPE"), (dict(h=250), "MLP_ESHAPE"),
                     (dict(s=0), "MLP_EINVAL"), (dict(X=None), "MLP_EINVAL"),
                     (dict(QKV=buf["QKV"].data_ptr() + 2), "MLP_EALIGN")):
        with pytest.raises(_lib.MlpError) as ei:
            fwd(**kw)
        assert ei.value.name == name, kw
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_attn_backward(dev["X"], dev["Wqkv"], dev["Wo"], buf["QKV"], buf["C"], buf["L"], dev["dY"], b, s, h,
                                  a, D, 1, True, buf["dX"], buf["dWqkv"], buf["dWo"], buf["ws"], buf["ws"].numel() - 256)
    assert ei.value.name == "MLP_EWORKSPACE"
    assert _lib.mlp_tp_attn_workspace_bytes(b, s, h, a, 64, 1) == 0


@pytest.mark.parametrize("name", ["gpt3-175b-attn", "gpt-18b-attn"])
def test_full_size_sampled(name):
    """The full-size workload in the bench's configuration: sampled C and L entries against
    the oracle, every output finite, and a second step bitwise equal to the first."""
    w = ATTN_WORKLOADS[name]
    inp = make_attn_workload_inputs(w)
    buf = _run(inp, w.b, w.s, w.a, w.t, w.causal)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(w.T, 14, replace=False), [0, w.s - 1, w.s, w.T - 1]]))
    heads = np.array([0, 37 % w.a, w.a - 1])
    C = buf["C"].view(w.T, w.a, D)[torch.from_numpy(rows).cuda()][:, torch.from_numpy(heads).cuda()].cpu()
    L = buf["L"].view(w.b, w.a, w.s)
    hsel = torch.from_numpy(heads).cuda()
    Lg = torch.stack([L[r // w.s, hsel, r % w.s] for r in rows.tolist()]).cpu()
    first = {k: buf[k].clone() for k in ("Y", "dX", "dWqkv", "dWo")}
    for k, v in first.items():
        assert torch.isfinite(v.float()).all(), k
    dev = {k: v.cuda() for k, v in inp.items()}
    block.attn_step(dev, buf, w.b, w.s, w.a, w.t, w.causal)
    for k, v in first.items():
        assert torch.equal(v, buf[k]), k
    del buf, first, dev
    gc.collect()
    torch.cuda.empty_cache()
    ref = oracle.attn_sampled_bf16(inp, w.b, w.s, w.a, rows, heads, w.causal)
    _close("C sampled", C, ref["C"])
    _close("L sampled", Lg, ref["L"])
